"""GB300-native hyper-connection mix statistics (hc_mix) for sm_103a.

The compute path is the C-ABI library libhcmix.so (hand-written CUDA kernels);
`hyper_connection_mix_gb300.binding` marshals arguments to it.  Importing this
package does not load the library; the first call into `binding` does, and it
raises if the library is missing -- there is no CPU fallback.
"""
__all__ = ["binding", "traffic"]
