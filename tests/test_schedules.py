"""Host-side checks of the library's schedules (no GPU): the work lists come
from the C ABI (bakron_schedule_export), the checks from the method.

Two-sided solve (summary page "FastKron: Efficient Quantization with
Kronecker-Factored Hessians", the derivation of BaKron-antidiagonal and of the
divide and conquer over anti-diagonals): the error of tile (I, J) reaches every
tile (I', J') with I' >= I, J' >= J through the row accumulator
R[I][J'] = sum_J E[I][J] U_A[J][J'] (stage 1 adds row updates into R, which
lives for the whole solve) and W~[I'][J'] -= U_B[I][I']^T R[I][J'] (stage 2,
R complete for I < I', R over J < J' for I = I').  The schedule must apply
each (source, target) contribution exactly once, from a source whose leaf has
run, before the leaf of the target: pairs on neighbouring tile diagonals
through the near products issued between the two leaves, every other pair
through a propagation that starts after the leaf of its last source.
One-sided solve (B = I): the same over column tiles.
Preparation: the blocked Cholesky's trailing updates and the
recursive-doubling inverse.

The stream model mirrors the executor's rules in csrc/api.cu: leaves and near
products on the critical stream; a propagation's chunks on its lane's urgent,
middle or lowest-priority stream by their slack, each stream starting after
the near products' stage 1 before the propagation; every chunk's stage 1
after the chunks enqueued earlier that write R tiles of the same diagonals,
its stage 2 after those that update W~ tiles of the same diagonals (a chunk
with both stages launches them together, after both kinds), and every
near product after both kinds for its diagonal, every leaf after the W~
updates of its diagonal.  The checks then require every update of a W~ or an
R tile (so their fp32 order is fixed) to form one chain, every R tile's
readers to sit between the writers enqueued before and after them, and every
E tile's producer and readers to be ordered by stream order and events.
"""

import numpy as np
import pytest

from kronecker_factored_gptq_gb300 import bakron as kb


def parse_solve(a):
    n_ops, n_chunks, n_items = (int(x) for x in a[:3])
    p = 3
    ops = a[p:p + 7 * n_ops].reshape(n_ops, 7); p += 7 * n_ops
    chunks = a[p:p + 6 * n_chunks].reshape(n_chunks, 6); p += 6 * n_chunks
    items = a[p:p + 4 * n_items].reshape(n_items, 4); p += 4 * n_items
    assert p == len(a)
    return ops, chunks, items


def parse_prepare(a):
    nb, n_items, n_levels = (int(x) for x in a[:3])
    p = 3
    syrk = a[p:p + 3 * nb].reshape(nb, 3); p += 3 * nb
    levels = []
    for _ in range(n_levels):
        n = int(a[p]); p += 1
        levels.append(a[p:p + 4 * n].reshape(n, 4)); p += 4 * n
    items = a[p:p + 4 * n_items].reshape(n_items, 4); p += 4 * n_items
    assert p == len(a)
    return syrk, levels, items


class Streams:
    """Happens-before over nodes enqueued on streams with events."""

    def __init__(self):
        self.anc = []          # ancestor bitmask per node
        self.last = {}         # stream -> last node
        self.pending_waits = {}

    def node(self, stream):
        m = 0
        if stream in self.last:
            p = self.last[stream]
            m |= self.anc[p] | (1 << p)
        for p in self.pending_waits.pop(stream, []):
            m |= self.anc[p] | (1 << p)
        self.anc.append(m)
        i = len(self.anc) - 1
        self.last[stream] = i
        return i

    def record(self, stream):
        """An event recorded now on `stream`: the node it completes after
        (a marker node when waits were enqueued after the last node)."""
        if self.pending_waits.get(stream):
            self.node(stream)
        return self.last.get(stream)

    def wait(self, stream, ev):
        if ev is not None:
            self.pending_waits.setdefault(stream, []).append(ev)

    def before(self, a, b):
        return bool((self.anc[b] >> a) & 1)


MID_SLACK = 15   # the executor's middle-priority bound (csrc/api.cu, kMidSlack)
FUSE_CLASS = 2   # classes whose chunks launch both stages together (kFuseClass)


def model_solve(ops, chunks, items, one_sided=False, wait_at_propagation=True):
    """Builds the stream model and returns (S, accesses) where accesses maps
    ('W', tile) / ('R', tile) / ('E', tile) to [(node, 'r'|'w')].  With
    wait_at_propagation False, propagation chunks skip the waits for earlier
    chunks of the same diagonals (the sensitivity check)."""
    S = Streams()
    acc = {}

    def touch(key, node, mode):
        acc.setdefault(key, []).append((node, mode))

    pending = []    # W~ writers: (event node, dlo, dhi)
    rpending = []   # R writers

    crit_waited = set()   # events the critical stream already waited for

    def order_before(lst, stream, lo, hi):
        keep = []
        for ev, dlo, dhi in lst:
            overlap = dlo < hi and dhi > lo
            if overlap and not (stream == "cs" and ev in crit_waited):
                S.wait(stream, ev)
                if stream == "cs":
                    crit_waited.add(ev)
            if not (overlap and lo <= dlo and dhi <= hi):
                keep.append((ev, dlo, dhi))
        lst[:] = keep

    def stage1(stream, its, n=None):
        n = S.node(stream) if n is None else n
        for Jp, I, k0, k1 in its:
            touch(("R", (I, Jp)), n, "w")   # read-modify-write of the fp32 sums
            for J in range(k0, k1):
                touch(("E", (I, J)), n, "r")
        return n

    def stage2(stream, its, n=None):
        n = S.node(stream) if n is None else n
        for Ip, Jp, k0, k1 in its:
            touch(("W", (Ip, Jp)), n, "w")
            for I in range(k0, k1):
                if one_sided:
                    touch(("E", (Ip, I)), n, "r")
                else:
                    touch(("R", (I, Jp)), n, "r")
        return n

    ev_leaf = None
    ev_near1 = None
    for kind, D, I0, ntiles, depth, chunk0, nchunks in ops.tolist():
        if kind == 0:
            order_before(pending, "cs", D, D + 1)
            n = S.node("cs")
            if one_sided:
                tiles = [(I, D) for I in range(ntiles)]
            else:
                tiles = [(I0 + t, D - I0 - t) for t in range(ntiles)]
            for t in tiles:
                touch(("W", t), n, "w")   # reads W~, the last of its updates
                touch(("E", t), n, "w")
            ev_leaf = S.record("cs")
            continue
        if kind == 2:
            dlo, dhi, off1, n1, off, nn = chunks[chunk0].tolist()
            order_before(rpending, "cs", D, D + 1)
            order_before(pending, "cs", D, D + 1)
            if n1 > 0:
                stage1("cs", items[off1:off1 + n1].tolist())
            ev_near1 = S.record("cs")
            if nn > 0:
                stage2("cs", items[off:off + nn].tolist())
            continue
        if one_sided:
            # one-sided path: first chunk on the critical stream, waits for the
            # deferred chunks of the same columns before it
            if wait_at_propagation and nchunks > 0:
                order_before(pending, "cs", chunks[chunk0][0], chunks[chunk0 + nchunks - 1][1])
            for c in range(nchunks):
                dlo, dhi, off1, n1, off, nn = chunks[chunk0 + c].tolist()
                stream = "cs" if c == 0 else "side%d" % depth
                if c == 1:
                    S.wait(stream, S.record("cs"))
                if nn > 0:
                    stage2(stream, items[off:off + nn].tolist())
                if c > 0:
                    pending.append((S.record(stream), dlo, dhi))
            continue
        # the chunk's stream by its slack (leaves between the propagation's
        # start, after leaf D, and its first target), as the executor does
        started = set()

        def stream_for(h, k):
            name = ["urg", "mid", "side"][k] + "%d" % depth
            if name not in started:
                S.wait(name, ev_near1)
                started.add(name)
            return name

        for c in range(nchunks):
            dlo, dhi, off1, n1, off, nn = chunks[chunk0 + c].tolist()
            slack = dlo - D - 1
            k = 0 if slack <= 1 else (1 if slack <= MID_SLACK else 2)
            if k <= FUSE_CLASS and n1 > 0 and nn > 0:
                # one launch holds both stages: one node touching both lists
                stream = stream_for(0, k)
                if wait_at_propagation:
                    order_before(rpending, stream, dlo, dhi)
                    order_before(pending, stream, dlo, dhi)
                node = S.node(stream)
                stage1(stream, items[off1:off1 + n1].tolist(), node)
                stage2(stream, items[off:off + nn].tolist(), node)
                ev = S.record(stream)
                rpending.append((ev, dlo, dhi))
                pending.append((ev, dlo, dhi))
                continue
            if n1 > 0:
                stream = stream_for(0, k)
                if wait_at_propagation:
                    order_before(rpending, stream, dlo, dhi)
                stage1(stream, items[off1:off1 + n1].tolist())
                rpending.append((S.record(stream), dlo, dhi))
            if nn > 0:
                stream = stream_for(1, k)
                if wait_at_propagation:
                    order_before(pending, stream, dlo, dhi)
                stage2(stream, items[off:off + nn].tolist())
                pending.append((S.record(stream), dlo, dhi))
    return S, acc


def ordering_violations(S, acc):
    bad = []
    for key, lst in acc.items():
        lst = sorted(set(lst))
        writers = [n for n, m in lst if m == "w"]
        if key[0] in ("W", "R"):
            # every read-modify-write of a W~ tile (updates and the leaf) or
            # of an R tile (row updates) in one chain
            for a_, b_ in zip(writers, writers[1:]):
                if not S.before(a_, b_):
                    bad.append((key, a_, b_))
        if key[0] != "W":
            # each reader after the latest writer enqueued before it, and
            # before the next writer
            for n, m in lst:
                if m != "r":
                    continue
                prev = [w for w in writers if w < n]
                nxt = [w for w in writers if w > n]
                if not prev or not S.before(prev[-1], n):
                    bad.append((key, "read before write", n))
                if nxt and not S.before(n, nxt[0]):
                    bad.append((key, "overwritten before read", n))
    return bad


def contributions_solve(ops, chunks, items, M, N):
    """count[Ip, Jp, I, J]: times the error of tile (I, J) reaches (Ip, Jp),
    following the row accumulators in the order the schedule lists their
    updates and reads (the stream model checks that execution keeps that
    order); also checks each product's sources are finished, its outputs lie
    in its chunk's range and its targets are not."""
    count = np.zeros((M, N, M, N), dtype=np.int32)
    rsum = {}        # R tile (I, J') -> source columns J added so far
    last_leaf = -1   # leaves run in diagonal order
    for kind, D, a2, a3, depth, chunk0, nchunks in ops.tolist():
        if kind == 0:
            assert D == last_leaf + 1
            last_leaf = D
            continue
        if kind == 2:
            assert D == last_leaf + 1, "near products run right before their leaf"
            assert nchunks == 1
        else:
            assert D == last_leaf, "a propagation starts right after its last source's leaf"
            s0, s1 = a2, a3
            assert s1 == D + 1
        for c in range(nchunks):
            dlo, dhi, off1, n1, off, nn = chunks[chunk0 + c].tolist()
            if kind == 2:
                assert (dlo, dhi) == (D, D + 1)
            seen = set()
            for Jp, I, k0, k1 in items[off1:off1 + n1].tolist():
                assert (I, Jp) not in seen, "R tile updated twice in one launch"
                seen.add((I, Jp))
                assert 0 <= k0 < k1 <= Jp + 1
                assert I + k1 - 1 <= last_leaf, "stage 1 reads an unfinished source"
                if kind == 1:
                    assert dlo <= I + Jp < dhi, "R tile outside its chunk's range"
                    assert s0 <= I + k0 and I + k1 - 1 < s1, "source outside the band"
                else:
                    assert I + Jp in (D - 1, D)
                rsum.setdefault((I, Jp), []).extend(range(k0, k1))
            for Ip, Jp, k0, k1 in items[off:off + nn].tolist():
                assert dlo <= Ip + Jp < dhi, "stage-2 target outside its chunk's range"
                assert Ip + Jp > last_leaf, "stage 2 updates a finished tile"
                assert 0 <= k0 < k1 <= Ip + 1
                for I in range(k0, k1):
                    if kind == 1:
                        assert s0 <= I + Jp < s1, "pushed R tile outside the band"
                    for J in rsum.get((I, Jp), []):
                        count[Ip, Jp, I, J] += 1
    return count


def expected_counts(M, N):
    I = np.arange(M)[:, None, None, None]
    J = np.arange(N)[None, :, None, None]
    i = np.arange(M)[None, None, :, None]
    j = np.arange(N)[None, None, None, :]
    return ((i <= I) & (j <= J) & ~((i == I) & (j == J))).astype(np.int32)


SHAPES = [(1, 1), (1, 6), (6, 1), (2, 3), (4, 4), (5, 9), (8, 8), (11, 6), (16, 13)]


@pytest.mark.parametrize("M,N", SHAPES)
def test_solve_schedule_applies_every_contribution_once(M, N):
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, M, N))
    leaves = [int(op[1]) for op in ops if op[0] == 0]
    assert leaves == list(range(M + N - 1)), "one leaf per tile anti-diagonal, in order"
    for op in ops:
        if op[0] == 0:
            D, I0, nt = int(op[1]), int(op[2]), int(op[3])
            assert I0 == max(0, D - N + 1) and I0 + nt - 1 == min(D, M - 1)
    count = contributions_solve(ops, chunks, items, M, N)
    np.testing.assert_array_equal(count, expected_counts(M, N))


@pytest.mark.parametrize("M,N", [(64, 64), (32, 112), (112, 32)])
def test_solve_schedule_full_size_shapes(M, N):
    """The 8192 x 8192 and the 4096 x 14336 / 14336 x 4096 workloads' tile
    grids: every contribution exactly once, before its target's leaf."""
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, M, N))
    count = contributions_solve(ops, chunks, items, M, N)
    np.testing.assert_array_equal(count, expected_counts(M, N))


@pytest.mark.parametrize("M,N", SHAPES + [(64, 64), (32, 112), (112, 32)])
def test_solve_schedule_executes_each_product_once(M, N):
    """No redundant tile products: with the row accumulators kept for the
    whole solve, each row update E[I,J] U_A[J,J'] (J <= J', the own term
    J = J' only where a row below reads it) and each push U_B[I,I']^T R[I,J']
    (I <= I', the diagonal-block term I = I' only for J' >= 1) is one 128^3
    product, so the K tiles of all items add up to
    M N (N + 1) / 2 - N + N M (M + 1) / 2 - M = M N (M + N) / 2 + M N - M - N,
    the method's m n (m + n) count at tile granularity plus the diagonal
    blocks."""
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, M, N))
    total = 0
    for dlo, dhi, off1, n1, off, nn in chunks.tolist():
        total += int(np.sum(items[off1:off1 + n1, 3] - items[off1:off1 + n1, 2]))
        total += int(np.sum(items[off:off + nn, 3] - items[off:off + nn, 2]))
    assert total == M * N * (M + N) // 2 + M * N - M - N


@pytest.mark.parametrize("M,N", SHAPES + [(64, 64), (32, 112)])
def test_solve_streams_order_every_tile_access(M, N):
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, M, N))
    S, acc = model_solve(ops, chunks, items)
    assert ordering_violations(S, acc) == []


def test_solve_streams_without_the_propagation_wait_overlap():
    """The checker is sensitive: without the waits of a propagation chunk for
    the earlier chunks of the same diagonals, two propagations can update the
    same W~ tiles, or the same row accumulator tiles, concurrently.  The
    stage-2 updates are atomic adds, so for W~ that was correct but the order
    of the adds, and with it the fp32 rounding, could change from run to run;
    the row accumulators are read-modify-written and need the order outright.
    Ordered updates make the solve bit-reproducible."""
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, 8, 8))
    S, acc = model_solve(ops, chunks, items, wait_at_propagation=False)
    bad = ordering_violations(S, acc)
    assert bad and {b[0][0] for b in bad} <= {"W", "R"}


@pytest.mark.parametrize("M,N", [(9, 7), (4, 4), (16, 13)])
def test_solve_near_products_reach_a_fixed_depth(M, N):
    """The near products issued between leaf D - 1 and leaf D read the
    diagonals D - h .. D - 1 (h the same for every D) and update the W~ tiles
    of diagonal D only; every propagation's sources are at least h + 1
    diagonals before its
    first target, so it can start h leaves early; no propagation sits
    between two leaves on the critical stream."""
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_SOLVE, M, N))
    crit = [int(k) for k in ops[:, 0] if k != 1]
    assert crit == [0] + [2, 0] * (M + N - 2)
    depth = set()
    for kind, D, _, _, _, chunk0, nchunks in ops.tolist():
        if kind != 2:
            continue
        dlo, dhi, off1, n1, off, nn = chunks[chunk0].tolist()
        src = [I + J for Jp, I, k0, k1 in items[off1:off1 + n1].tolist() for J in range(k0, k1)]
        assert src and max(src) <= D - 1
        depth.add(D - min(src))
        for Ip, Jp, k0, k1 in items[off:off + nn].tolist():
            assert Ip + Jp == D
    h = max(depth)
    assert h >= 1 and all(d == min(h, D) for d, D in zip(sorted(depth), sorted(depth)))
    for kind, D, s0, s1, _, chunk0, nchunks in ops.tolist():
        if kind == 1:
            assert all(int(chunks[chunk0 + c][0]) >= s1 + h for c in range(nchunks))


@pytest.mark.parametrize("M,N", [(1, 1), (3, 1), (1, 7), (4, 5), (9, 16), (6, 33), (64, 64), (32, 112)])
def test_rows_schedule(M, N):
    ops, chunks, items = parse_solve(kb.schedule_export(kb.SCHEDULE_ROWS, M, N))
    assert [int(op[1]) for op in ops if op[0] == 0] == list(range(N))
    # exactly-once: column tile J reaches J' > J for every row tile, before leaf J'
    count = np.zeros((M, N, N), dtype=np.int32)   # [row, target J', source J]
    done = set()
    for kind, J, _, _, depth, chunk0, nchunks in ops:
        if kind == 0:
            done.add(J)
            continue
        for c in range(nchunks):
            dlo, dhi, off1, n1, off, nn = chunks[chunk0 + c]
            assert n1 == 0
            for I, Jp, k0, k1 in items[off:off + nn]:
                assert dlo <= Jp < dhi
                for Js in range(k0, k1):
                    assert Js in done and Js < Jp
                    count[I, Jp, Js] += 1
    want = np.broadcast_to(np.tril(np.ones((N, N), dtype=np.int32), -1), (M, N, N))
    np.testing.assert_array_equal(count, want)
    S, acc = model_solve(ops, chunks, items, one_sided=True)
    assert ordering_violations(S, acc) == []


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 8, 13, 17, 64, 112])
def test_prepare_trailing_updates_once_in_groups(nb):
    """Right-looking blocked Cholesky: every trailing tile (r, c) receives
    every panel j < c exactly once, after panel j is done (step >= j) and
    before the chain needs the tile (the step that reads column c is c - 1:
    the urgent tile and the lookahead group of step j are exactly what
    steps j + 1 and j + 2 read).  Panels reach a far tile singly or in a
    batch of consecutive panels (one product over their K range), applied
    at a step >= the batch's last panel and at least two steps before the
    tile's column is read."""
    syrk, levels, items = parse_prepare(kb.schedule_export(kb.SCHEDULE_PREPARE, nb))
    seen = {}
    for j in range(nb):
        off, n1, n2 = (int(x) for x in syrk[j])
        grp = [items[off:off + 1] if j + 1 < nb else items[off:off]]
        grp.append(items[off + 1:off + 1 + n1])
        grp.append(items[off + 1 + n1:off + 1 + n1 + n2])
        urgent, s1 = ({(int(r), int(c)) for r, c, k0, k1 in g} for g in grp[:2])
        for gi, g in enumerate(grp):
            for r, c, k0, k1 in g.tolist():
                assert 0 <= k0 < k1 <= j + 1, "a panel that is not done yet"
                if gi < 2:
                    assert (k0, k1) == (j, j + 1), "one panel per urgent / lookahead update"
                else:
                    assert k1 - k0 == 1 or k1 == j + 1, "a batch ends with this step's panel"
                    assert c - 1 >= j + 2 or k1 - k0 == 1, "a batched tile is read two steps later"
                for p in range(k0, k1):
                    key = (r, c, p)
                    assert key not in seen, key
                    seen[key] = True
        assert urgent == ({(j + 1, j + 1)} if j + 1 < nb else set())
        want1 = {(r, j + 1) for r in range(j + 2, nb)} | ({(j + 2, j + 2)} if j + 2 < nb else set())
        assert s1 == want1
        # the bulk group never touches what the urgent or lookahead groups of
        # this step hold, nor a column the chain already passed
        for r, c, k0, k1 in grp[2].tolist():
            assert c >= j + 2 and (r, c) != (j + 2, j + 2)
    want = {(r, c, j) for c in range(nb) for r in range(c, nb) for j in range(c)}
    assert set(seen) == want


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 6, 8, 11, 16, 64])
def test_prepare_doubling_inverts_a_block_triangle(nb):
    """Run the doubling pairs level by level on a random lower-triangular G of
    nb 3 x 3 blocks (T = (G21 Ginv11)^T, then Ginv21 = -Ginv22 T^T with its
    transposed copy): the result is G^{-1}."""
    _, levels, items = parse_prepare(kb.schedule_export(kb.SCHEDULE_PREPARE, nb))
    b = 3
    n = nb * b
    rng = np.random.default_rng(nb)
    G = np.tril(rng.standard_normal((n, n))) + 4 * np.eye(n)

    def t(X, r, c):
        return X[r * b:(r + 1) * b, c * b:(c + 1) * b]

    Gi = np.full((n, n), np.nan)
    GiT = np.full((n, n), np.nan)
    T = np.full((n, n), np.nan)
    for i in range(nb):
        for j in range(nb):
            if j > i:
                t(Gi, i, j)[:] = 0.0
                t(GiT, j, i)[:] = 0.0
        x = np.linalg.inv(t(G, i, i))
        t(Gi, i, i)[:] = x
        t(GiT, i, i)[:] = x.T
    assert len(levels) == max(0, int(np.ceil(np.log2(nb))))
    for pairs in levels:
        for t_off, t_n, x_off, x_n in pairs:
            for r, c, k0, k1 in items[t_off:t_off + t_n]:
                t(T, r, c)[:] = sum(t(GiT, r, k) @ t(G, c, k).T for k in range(k0, k1))
            for r, c, k0, k1 in items[x_off:x_off + x_n]:
                x = -sum(t(Gi, r, k) @ t(T, c, k).T for k in range(k0, k1))
                t(Gi, r, c)[:] = x
                t(GiT, c, r)[:] = x.T
    assert np.all(np.isfinite(Gi))
    np.testing.assert_allclose(Gi @ G, np.eye(n), atol=1e-12)
    np.testing.assert_array_equal(GiT, Gi.T)


def test_schedule_export_rejects_bad_arguments():
    import ctypes
    L = kb.lib()
    n = ctypes.c_int64(0)
    for args in ((0, 0, 4), (0, 4, 0), (1, 8193, 1), (2, 0, 1), (9, 2, 2)):
        assert L.bakron_schedule_export(args[0], args[1], args[2], None, 0, ctypes.byref(n)) == 1
    assert L.bakron_schedule_export(0, 4, 4, None, 0, None) == 1
    # a buffer smaller than the schedule is left untouched
    need = ctypes.c_int64(0)
    assert L.bakron_schedule_export(0, 3, 3, None, 0, ctypes.byref(need)) == 0
    buf = (ctypes.c_int32 * 4)(-7, -7, -7, -7)
    assert L.bakron_schedule_export(0, 3, 3, buf, 4, ctypes.byref(n)) == 0
    assert n.value == need.value and list(buf) == [-7, -7, -7, -7]
