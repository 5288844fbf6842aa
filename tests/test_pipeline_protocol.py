"""The tensor-core kernel's hand-off protocol, checked on the CPU.

The kernel's roles (x producer, two halves of four transform warps, four MMA
issuers, four accumulate warps, the W-slot refills) hand chunks to each other
through mbarriers whose waits only test the parity of the phase they want.
Such a wait is sound only when the waiter already knows the phase before it
complete; otherwise it cannot tell phase p - 2 from phase p and returns early.
This module restates, role by role, the waits and arrivals of
hyper_connection_mix_gb300/csrc/hcmix_tc.cuh as a model with real parity
semantics (the barrier's phase counter, arrival counts, a wait that returns
when the current phase parity differs), runs it under random interleavings
with the MMAs completing in issue order and the x loads landing in any order,
and asserts for every wait that the exact phase it needed had completed, and
that every run finishes.  It is a model of the kernel's protocol, kept beside
the kernel; the GPU tests check the kernel itself.
"""
import random

import pytest

X_STAGES, N_A, N_D, N_SQ, SLOTS, N_MMA = 3, 2, 4, 8, 2, 4
SHARED_A_EMPTY = False  # a planted mistake for the test that checks the model has teeth


class Bar:
    def __init__(self, count, name):
        self.count, self.pending, self.phase, self.name = count, count, 0, name

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than expected"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


def run_cta(u_begin, n, n_tiles, seed, packed=False):
    """One CTA's units [u_begin, u_begin + n) of a grid with n_tiles tiles per
    slice.  Returns the list of aliasing errors (empty when sound); raises on a
    deadlock."""
    rnd = random.Random(seed)
    sl = [(u_begin + i) // n_tiles for i in range(n)]
    s_first = sl[0]
    n_sl = sl[-1] - s_first + 1
    nck, nld = 4 * n, 2 * n
    mk = lambda p, c, m: [Bar(c, f"{p}{i}") for i in range(m)]
    full_x, empty_x = mk("full_x", 1, X_STAGES), mk("empty_x", 8, X_STAGES)
    # mma_ready[k % 4]: the transform warps of chunk k (4) and the accumulate
    # warps once they have read chunk k - 4 (4; made at set-up for k < 4)
    mma_ready, a_empty = mk("mma_ready", 8, N_D), mk("a_empty", 1, N_A)
    for b in mma_ready:
        for _ in range(4):
            b.arrive()
    sq_full, chunk_done = mk("sq_full", 4, N_SQ), mk("chunk_done", 4, N_SQ)
    d_full, w_full = mk("d_full", 1, N_D), mk("w_full", 1, 4 * SLOTS)
    dconv = Bar(4, "dconv")
    errors, pipe, tma = [], [], []

    def wait(bar, phase, who):
        parity = phase & 1
        while (bar.phase & 1) == parity:
            yield (bar, parity)
        if bar.phase <= phase:
            errors.append(f"{who}: {bar.name} wanted phase {phase}, barrier at {bar.phase}")

    def x_producer():
        for L in range(nld):
            st = L % X_STAGES
            if L >= X_STAGES:
                yield from wait(empty_x[st], L // X_STAGES - 1, f"x L{L}")
            tma.append(st)
            yield None

    def transform(h, q):
        for L in range(nld):
            k, st = 2 * L + h, L % X_STAGES
            yield from wait(full_x[st], L // X_STAGES, f"T{h}{q} k{k} x")
            yield None
            empty_x[st].arrive()
            if k >= N_SQ:
                yield from wait(chunk_done[k % N_SQ], k // N_SQ - 1, f"T{h}{q} k{k} sq")
            sq_full[k % N_SQ].arrive()
            if k >= N_A:  # A buffer h, last used by chunk k - 2
                if SHARED_A_EMPTY:  # planted: one barrier for both halves' chunks
                    yield from wait(a_empty[0], k - 2, f"T{h}{q} k{k} A")
                else:
                    yield from wait(a_empty[h], k // N_A - 1, f"T{h}{q} k{k} A")
            yield None
            mma_ready[k % N_D].arrive()

    def issuer(c):  # chunk c of every unit
        prev = -1
        for i in range(n):
            k = 4 * i + c
            s = sl[i]
            j = s - s_first
            first = s != prev
            prev = s
            yield from wait(mma_ready[c], i, f"I{c} k{k} ready")
            if first:
                yield from wait(w_full[(j % SLOTS) * 4 + c], j // SLOTS, f"I{c} k{k} W")
            yield None
            pipe.append(k)

    def accumulate(q):
        if not packed and n_sl >= 2:  # the second slice, converted during set-up
            yield None
            dconv.arrive()
            while dconv.phase == 0:
                yield (dconv, 0)
            if q == 0:
                for c in range(4):
                    w_full[4 + c].arrive()
        for k in range(nck):
            yield from wait(d_full[k % N_D], k // N_D, f"D{q} k{k}")
            yield from wait(sq_full[k % N_SQ], k // N_SQ, f"D{q} k{k} sq")
            yield None
            chunk_done[k % N_SQ].arrive()
            mma_ready[k % N_D].arrive()  # D buffer k % 4 free for chunk k + 4
            i = k // 4
            if k % 4 == 3:
                j = sl[i] - s_first
                if j + SLOTS < n_sl and (i == n - 1 or sl[i + 1] != sl[i]) and q == 0:
                    for c in range(4):  # refill: slice j + 2 into slot j % 2
                        w_full[((j + SLOTS) % SLOTS) * 4 + c].arrive()

    for c in range(4 * min(SLOTS, n_sl) if packed else 4):
        w_full[c].arrive()  # set-up: the first slice (and the second, prepacked)
    roles = {"x": x_producer()}
    roles.update({f"I{g}": issuer(g) for g in range(N_MMA)})
    roles.update({f"T{h}{q}": transform(h, q) for h in (0, 1) for q in range(4)})
    roles.update({f"D{q}": accumulate(q) for q in range(4)})
    state = {r: None for r in roles}
    done = set()
    while True:
        ready = [r for r in roles if r not in done and
                 (state[r] is None or (state[r][0].phase & 1) != state[r][1])]
        if (pipe or tma) and (not ready or rnd.random() < 0.3):
            if pipe and (not tma or rnd.random() < 0.5):
                k = pipe.pop(0)  # the tensor pipe completes MMAs in issue order
                d_full[k % N_D].arrive()
                a_empty[0 if SHARED_A_EMPTY else k % N_A].arrive()
            else:
                full_x[tma.pop(rnd.randrange(len(tma)))].arrive()
            continue
        if not ready:
            assert len(done) == len(roles), \
                f"deadlock: {[(r, state[r][0].name) for r in roles if r not in done]}"
            return errors
        r = rnd.choice(ready)
        try:
            state[r] = next(roles[r])
        except StopIteration:
            done.add(r)


def grid_ctas(M, K, sms=152):
    n_tiles = (M + 127) // 128
    U = n_tiles * (K // 256)
    G = min(sms, U)
    return [(b * U // G, (b + 1) * U // G - b * U // G, n_tiles) for b in range(G)]


@pytest.mark.parametrize("M,K", [(1, 20480), (4096, 20480), (512, 20480), (130, 131072),
                                 (5, 131072), (256, 65536)])
def test_protocol_sound_and_deadlock_free(M, K):
    ctas = grid_ctas(M, K)
    # every distinct CTA shape (units, slice boundaries relative to the range)
    shapes = {}
    for ub, n, nt in ctas:
        key = (n, tuple((ub + i) // nt - ub // nt for i in range(n)))
        shapes.setdefault(key, (ub, n, nt))
    for ub, n, nt in shapes.values():
        for seed in range(6):
            for packed in (False, True):
                errs = run_cta(ub, n, nt, seed, packed)
                assert not errs, f"M={M} K={K} units {ub}+{n} seed {seed}: {errs[:3]}"


def test_model_catches_an_unordered_parity_wait():
    """The check has teeth: with one a_empty barrier shared by both halves of
    the transform warps (each half then sees only every other phase) the model
    reports an early return or the deadlock it leads to."""
    global SHARED_A_EMPTY
    SHARED_A_EMPTY = True
    found = False
    try:
        for ub, n, nt in grid_ctas(4096, 20480)[:8]:
            for seed in range(8):
                try:
                    found = found or bool(run_cta(ub, n, nt, seed))
                except AssertionError:
                    found = True
    finally:
        SHARED_A_EMPTY = False
    assert found
