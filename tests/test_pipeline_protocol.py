"""The tensor-core kernel's hand-off protocol, checked on the CPU.

The kernel's roles (the x producer, three thirds of four transform warps by
chunk, three MMA issuers, two halves of four accumulate warps by unit, the
W-slot refills) hand chunks to each other through mbarriers whose waits only test the
parity of the phase they want; the chunk's sum of squares travels in a TMEM
column (k % 6) written with the chunk's A and read with its D, guarded by no
barrier of its own.  Such a wait is sound only when the waiter
already knows the phase before it complete; otherwise it cannot tell phase
p - 2 from phase p and returns early.  This module restates, role by role, the
waits and arrivals of hyper_connection_mix_gb300/csrc/hcmix_tc.cuh as a model
with real parity semantics (the barrier's phase counter, arrival counts, a
wait that returns when the current phase parity differs), runs it under random
interleavings with the MMAs completing in issue order and the x loads landing
in any order, and asserts
  * for every wait, that the exact phase it needed had completed;
  * for every buffer (x stage, TMEM A and D buffers, sum-of-squares column,
    W slot), that it is only rewritten once every reader of its previous
    contents is done, and that the sum column read with chunk k's D holds
    chunk k's value;
  * that every run finishes.
It is a model of the kernel's protocol, kept beside the kernel; the GPU tests
check the kernel itself.
"""
import random

import pytest

X_STAGES, CPS, N_A, N_D, N_SQ, SLOTS, N_MMA = 6, 1, 3, 3, 6, 2, 3  # CPS: chunks per x stage
PLANTED = None  # a planted mistake for the tests that check the model has teeth


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
    slice.  Returns the list of errors (empty when sound); raises on a
    deadlock."""
    rnd = random.Random(seed)
    sl = [(u_begin + i) // n_tiles for i in range(n)]
    s_first = sl[0]
    n_sl = sl[-1] - s_first + 1
    nck, nld = 4 * n, 4 * n // CPS
    mk = lambda p, c, m: [Bar(c, f"{p}{i}") for i in range(m)]
    full_x, empty_x = mk("full_x", 1, X_STAGES), mk("empty_x", 4 * CPS, X_STAGES)
    # mma_ready[k % 3]: the four transform warps of chunk k and the four
    # accumulate warps that have read chunk k - 3 (made at set-up for k < 3)
    mma_ready = mk("mma_ready", 8, N_MMA)
    for b in mma_ready:
        for _ in range(4):
            b.arrive()
    # d_full[b * 2 + h]: D buffer b holds a chunk of accumulate half h
    d_full, w_full = mk("d_full", 1, 2 * N_D), mk("w_full", 1, 4 * SLOTS)
    dconv = Bar(8, "dconv")
    # refill_done[h]: the half's four warps have converted a refilled slot
    refill_done = mk("refill_done", 4, 2)
    errors, pipe, tma = [], [], []
    # progress, for the buffer checks
    x_read = [0] * nld          # transform warps that have read x load L
    mma_done = set()            # chunks whose MMAs completed
    d_read = [0] * nck          # accumulate warps that have read D of chunk k
    sq_read = [0] * nck         # accumulate warps that have read the sum of squares of chunk k
    sq_col = {}                 # (column, quadrant) -> the chunk whose sum it holds
    slice_done = set()          # slices whose every MMA completed (W slot free)
    converted = {}              # refilled slice -> warps of its half that have converted their share

    def wait(bar, phase, who):
        parity = phase & 1
        while (bar.phase & 1) == parity:
            yield (bar, parity)
        if bar.phase <= phase:
            errors.append(f"{who}: {bar.name} wanted phase {phase}, barrier at {bar.phase}")

    def check(cond, what):
        if not cond:
            errors.append(what)

    def issue_load(L):
        check(L < X_STAGES or x_read[L - X_STAGES] == 4 * CPS, f"x load {L} over an unread stage")
        tma.append((L % X_STAGES, L))

    def x_producer():  # the loads after the first (set-up issues load 0)
        for L in range(1, nld):
            if L >= X_STAGES:
                yield from wait(empty_x[L % X_STAGES], L // X_STAGES - 1, f"x L{L}")
            issue_load(L)
            yield None

    def transform(tt, q):  # the chunks k with k % 3 == tt
        ae_seen = [0, 0]  # phases of d_full[tt * 2 + h] waited for so far
        for k in range(tt, nck, N_A):
            L, st = k // CPS, (k // CPS) % X_STAGES
            s_ = k % (3 if PLANTED == "sq_col_mod3" else N_SQ)
            yield from wait(full_x[st], L // X_STAGES, f"T{tt}{q} k{k} x")
            yield None
            x_read[L] += 1
            empty_x[st].arrive()
            if k >= N_A:  # chunk k - 3 (this third's) is done with A buffer tt: its D commit
                h = ((k - N_A) // 4) % 2
                a = (tt + 1) % N_A if PLANTED == "wrong_a_buffer" else tt
                yield from wait(d_full[a * 2 + h], ae_seen[h], f"T{tt}{q} k{k} A")
                ae_seen[h] += 1
                check(k - N_A in mma_done, f"A buffer of chunk {k} rewritten before the MMAs of {k - N_A} were done")
            # the A limbs and the sum of squares into TMEM
            old = sq_col.get((s_, q))
            check(old is None or sq_read[old] == 4, f"sum column of chunk {k} over chunk {old}'s unread one")
            sq_col[(s_, q)] = k
            yield None
            mma_ready[k % N_MMA].arrive()

    def issuer(t):  # the chunks k with k % 3 == t
        for k in range(t, nck, N_MMA):
            i, c = divmod(k, 4)
            s = sl[i]
            j = s - s_first
            yield from wait(mma_ready[t], k // N_MMA, f"I{t} k{k} ready")
            # a W barrier: its earlier fill always completed before any issuer
            # waits for the next, so several issuers may wait on it
            yield from wait(w_full[(j % SLOTS) * 4 + c], j // SLOTS, f"I{t} k{k} W")
            check(k < N_D or d_read[k - N_D] == 4, f"D buffer of chunk {k} over an unread one")
            check(j < SLOTS or (s - SLOTS) in slice_done, f"chunk {k} reads a W slot being refilled")
            yield None
            pipe.append((k, (k % N_D) * 2 + i % 2))

    def accumulate(dh, q):  # the units i with i % 2 == dh, quadrant q
        if not packed:  # the first two slices' W, converted by all eight first
            for j in range(min(SLOTS, n_sl)):
                yield None
                dconv.arrive()
                while dconv.phase <= j:
                    yield (dconv, j & 1)
                if dh == 0 and q == 0:
                    for c in range(4):
                        w_full[4 * j + c].arrive()
        seen = [0] * N_D  # phases of d_full[b * 2 + dh] waited for so far
        rf_seen = 0  # phases of refill_done[dh] waited for so far (warp q == 0)
        for i in range(dh, n, 2):
            for c in range(4):
                k = 4 * i + c
                b = k % N_D
                dbar = b * 2 + dh if PLANTED != "d_full_by_buffer" else b * 2
                yield from wait(d_full[dbar], seen[b], f"D{dh}{q} k{k}")
                seen[b] += 1
                s_ = k % (3 if PLANTED == "sq_col_mod3" else N_SQ)
                check(k in mma_done, f"D of chunk {k} read before its MMAs completed")
                check(sq_col.get((s_, q)) == k, f"chunk {k} read its sum column holding chunk {sq_col.get((s_, q))}")
                yield None
                d_read[k] += 1
                sq_read[k] += 1
                mma_ready[b].arrive()  # D buffer b free for chunk k + 3
            j = sl[i] - s_first
            if j + SLOTS < n_sl and (i == n - 1 or sl[i + 1] != sl[i]):
                # refill: slice j + 2 into slot j % 2.  Converted in-kernel: every
                # warp of the half arrives on refill_done, the first waits there
                # and then marks the slot full; prepacked limbs: the first warp
                # issues the loads
                if not packed:
                    yield None
                    converted[j + SLOTS] = converted.get(j + SLOTS, 0) + 1
                    refill_done[dh].arrive()
                if q == 0:
                    if not packed and PLANTED != "refill_no_wait":
                        yield from wait(refill_done[dh], rf_seen, f"D{dh}{q} refill {j + SLOTS}")
                        rf_seen += 1
                    check(packed or converted.get(j + SLOTS) == 4,
                          f"slot of slice {j + SLOTS} marked full before its conversion was done")
                    slice_done.add(sl[i])
                    for c in range(4):
                        w_full[((j + SLOTS) % SLOTS) * 4 + c].arrive()

    if packed:
        for c in range(4 * min(SLOTS, n_sl)):
            w_full[c].arrive()  # set-up: TMA loads of the first two slices' limbs
    if nld:  # set-up: the first x load
        issue_load(0)
    roles = {"x": x_producer()}
    roles.update({f"I{g}": issuer(g) for g in range(N_MMA)})
    roles.update({f"T{t}{q}": transform(t, q) for t in range(N_A) for q in range(4)})
    roles.update({f"D{h}{q}": accumulate(h, q) for h in (0, 1) for q in range(4)})
    state = {r: None for r in roles}
    done = set()
    while True:
        ready = [r for r in roles if r not in done and
                 (state[r] is None or (state[r][0].phase & 1) != state[r][1])]
        if (pipe or tma) and (not ready or rnd.random() < 0.3):
            if pipe and (not tma or rnd.random() < 0.5):
                k, dbar = pipe.pop(0)  # the tensor pipe completes MMAs in issue order
                mma_done.add(k)
                d_full[dbar].arrive()
            else:
                st, _ = tma.pop(rnd.randrange(len(tma)))
                full_x[st].arrive()
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


def distinct_shapes(M, K):
    shapes = {}
    for ub, n, nt in grid_ctas(M, K):
        key = (n, tuple((ub + i) // nt - ub // nt for i in range(n)))
        shapes.setdefault(key, (ub, n, nt))
    return list(shapes.values())


@pytest.mark.parametrize("M,K", [(1, 20480), (4096, 20480), (512, 20480), (130, 131072),
                                 (5, 131072), (256, 65536)])
def test_protocol_sound_and_deadlock_free(M, K):
    # every distinct CTA shape (units, slice boundaries relative to the range)
    for ub, n, nt in distinct_shapes(M, K):
        for seed in range(6):
            for packed in (False, True):
                errs = run_cta(ub, n, nt, seed, packed)
                assert not errs, f"M={M} K={K} units {ub}+{n} seed {seed}: {errs[:3]}"


@pytest.mark.parametrize("mistake", ["wrong_a_buffer", "d_full_by_buffer", "refill_no_wait",
                                     "sq_col_mod3"])
def test_model_catches_planted_mistakes(mistake):
    """The checks have teeth: a transform third that waits on another third's
    A barrier, accumulate halves that share one D barrier per buffer (each
    then sees only some of its phases), a refilled W slot marked full by
    the half's first warp without waiting for the other three, or sum-of-
    squares columns reused every three chunks instead of six, are reported
    (an early return, a buffer rewritten or used too soon, or the deadlock
    they lead to)."""
    global PLANTED
    PLANTED = mistake
    found = False
    # the refill needs CTAs with more than two slices: M = 130, K = 131072
    ctas = grid_ctas(130, 131072)[:8] if mistake == "refill_no_wait" else grid_ctas(4096, 20480)[:8]
    try:
        for ub, n, nt in ctas:
            for seed in range(8):
                try:
                    found = found or bool(run_cta(ub, n, nt, seed))
                except AssertionError:
                    found = True
    finally:
        PLANTED = None
    assert found
