"""Host-side checks of bench.py's timing loop: exactly the requested number of
calls is replayed, whatever the graph size."""
import bench


class _Graph:
    def __init__(self):
        self.replays = 0

    def replay(self):
        self.replays += 1


def test_replay_calls_issues_exactly_k_calls():
    for k in (0, 1, 9, 10, 11, 20, 23, 20000):
        many, one = _Graph(), _Graph()
        bench.replay_calls((many, one), k)
        assert many.replays * bench.GRAPH_CALLS + one.replays == k
        assert one.replays < bench.GRAPH_CALLS


def test_protocols_flag_parses():
    assert bench.parse_args(["--protocols"]).protocols
    assert not bench.parse_args([]).protocols
