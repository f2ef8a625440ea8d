"""A host model of how the row pass cuts one row into groups, slices, chunks and direct loads.

The row pass (K1 / K1g) follows each target row's own 16-byte grid: the first H entries (the
head, before the row's first 16-byte boundary, H < 16 / element bytes) form group 0, read by
rank 0 with element loads; the body [H, V) is cut into 8-entry groups 1, 2, ... and into the
cluster's C slices of `slice` entries (a multiple of 8).  Inside a slice, whole chunks of 8-entry
groups go through the bulk-copy ring; what is left of the slice (fewer than 8 entries at its end)
and the head are direct loads, group g going to consumer thread g mod (consumer threads).

The model restates that arithmetic and checks, for every vocabulary size, cluster size, head
length and CTA shape listed, that every entry of the row is visited exactly once and that the
group it is visited in is the group the argmax re-read searches for it.  A plausible slip in
the kernel's index arithmetic (a slice boundary off by one group, the head counted twice, a
ragged end skipped) fails one of these cases.  It checks the partition, not the kernel: the GPU
parity tests check the kernel's outputs.
"""

import pytest


def slice_entries(V, C):
    per = (V + C - 1) // C
    return (per + 7) & ~7


def visit_row(V, C, head_offset_bytes, elem_bytes, chunk, consumers):
    H = min(((16 - head_offset_bytes % 16) % 16) // elem_bytes, V)
    Vb = V - H
    S = slice_entries(V, C)
    seen = {}
    for rank in range(C):
        vb = rank * S
        ve = min(Vb, vb + S)
        length = max(0, ve - vb)
        ngroups = (length + 7) >> 3
        body = length & ~7
        has_head = 1 if (rank == 0 and H > 0) else 0
        ngx = ngroups + has_head
        gfirst = 1 + (vb >> 3)
        for e0 in range(0, body, chunk):  # the ring's chunks
            for g in range(min(chunk, body - e0) >> 3):
                grp = gfirst + (e0 >> 3) + g
                for j in range(8):
                    seen.setdefault(H + vb + e0 + 8 * g + j, []).append(grp)
        for tid in range(consumers):  # direct loads: the ragged end, and the head on rank 0
            g = (body >> 3) + ((tid - (body >> 3)) & (consumers - 1))
            while g < ngx:
                head = g == ngroups
                v0 = 0 if head else H + vb + (g << 3)
                n = H if head else min(8, ve - (vb + (g << 3)))
                grp = 0 if head else gfirst + g
                for j in range(n):
                    seen.setdefault(v0 + j, []).append(grp)
                g += consumers
    assert sorted(seen) == list(range(V)), ("entries", V, C, head_offset_bytes, elem_bytes)
    for v, groups in seen.items():
        assert len(groups) == 1, ("visited twice", v)
        grp = groups[0]
        lo, n = (0, H) if grp == 0 else (H + 8 * (grp - 1), min(8, V - (H + 8 * (grp - 1))))
        assert lo <= v < lo + n, ("argmax re-read misses", v, grp)


# (entries per chunk, consumer threads): the forward for two 16-bit inputs, the pass with
# the gradient, and either one with a float32 input (half the entries per chunk)
SHAPES = [(8192, 256), (4096, 128), (4096, 256), (2048, 128)]


@pytest.mark.parametrize("elem_bytes", [2, 4])
def test_small_rows_every_cluster_and_head(elem_bytes):
    for V in range(1, 40):
        for C in range(1, 9):
            for off in range(0, 16, elem_bytes):
                for chunk, consumers in SHAPES:
                    visit_row(V, C, off, elem_bytes, chunk, consumers)


@pytest.mark.parametrize("V", [1001, 4097, 8200, 151936, 151937])
def test_large_rows(V):
    for C in (1, 2, 6, 8):
        for elem_bytes, offs in ((2, (0, 2, 14)), (4, (0, 4, 12))):
            for off in offs:
                for chunk, consumers in SHAPES[:2]:
                    visit_row(V, C, off, elem_bytes, chunk, consumers)


# ---------------------------------------------------------------------------------------------
# The second pass's reuse of the ring (the row pass with the gradient).
#
# Ring position cc (counted over the CTA's whole life) uses stage cc mod S.  A paired row queues
# its nch chunks twice: the first pass in order, then the second pass, whose first min(S, nch)
# positions take, when nch >= S, the first pass's last S chunks in ascending order without a copy
# (the stage still holds them), and whose other positions copy the remaining chunks last one
# first.  The first pass asks L2 to drop at once exactly the chunks the second pass takes from the
# ring.  The model replays that order over a sequence of units and checks that each reused stage
# still holds the chunk the second pass wants, that the second pass sees every chunk once, and that
# the early-drop set is the reused set.  A slip such as reusing when nch < S, or an off-by-one in
# the chunk a reused position maps to, fails it.


def second_pass_reuses(ci, nch, S):
    return nch >= S and ci < S


def second_pass_chunk(ci, nch, S):
    return nch - S + ci if second_pass_reuses(ci, nch, S) else nch - 1 - ci


def replay_ring(units, S):
    stage = [None] * S  # (unit, chunk) each stage holds
    cc = 0
    for u, (nch, passes) in enumerate(units):
        dropped_early = set()
        for ci in range(nch):  # first pass
            stage[cc % S] = (u, ci)
            if passes == 2 and nch >= S and ci >= nch - S:
                dropped_early.add(ci)
            cc += 1
        if passes == 1:
            continue
        seen, reused = [], set()
        for ci in range(nch):  # second pass
            want = second_pass_chunk(ci, nch, S)
            if second_pass_reuses(ci, nch, S):
                assert stage[cc % S] == (u, want), ("stage no longer holds the chunk", u, nch, S, ci)
                reused.add(want)
            else:
                stage[cc % S] = (u, want)
            seen.append(want)
            cc += 1
        assert sorted(seen) == list(range(nch)), ("second pass order", nch, S)
        assert reused == dropped_early, ("early drop set", nch, S)
        if nch >= S:  # the reused chunks come first, ascending
            assert seen[:S] == list(range(nch - S, nch))


@pytest.mark.parametrize("S", [3, 4])
def test_second_pass_reuse_of_the_ring(S):
    for nch in range(0, 14):
        replay_ring([(nch, 2)], S)
    import random
    rng = random.Random(5 + S)
    for _ in range(200):  # paired rows (two passes) and bonus rows (one) in any order
        replay_ring([(rng.randrange(0, 14), rng.choice((1, 2))) for _ in range(rng.randrange(1, 9))], S)


# ---------------------------------------------------------------------------------------------
# Unit order of the row pass with the gradient.  Units 0 .. N_d - 1 are the paired rows and
# N_d .. N_d + R - 1 the target-only rows; cluster cid takes positions cid, cid + ncl, ...  When
# one launch takes every unit, the first `early` = min(R, ncl // 4) positions hold target-only
# rows, then come all paired rows, then the remaining target-only rows.  The model checks that
# the order is a permutation (every row handled once), that exactly `early` clusters start with
# a target-only row, and that the paired rows keep their relative order.


def unit_at(u, N_d, R, ncl, whole_launch=True):
    early = min(R, ncl // 4) if whole_launch else 0
    return N_d + u if u < early else (u - early if u < N_d + early else u)


@pytest.mark.parametrize("N_d,R,ncl", [(914, 128, 97), (289, 32, 101), (8192, 512, 97), (16, 1, 152),
                                       (3, 3, 4), (0, 5, 8), (40, 0, 20), (5, 200, 64)])
def test_unit_order_is_a_permutation(N_d, R, ncl):
    n = N_d + R
    order = [unit_at(u, N_d, R, ncl) for u in range(n)]
    assert sorted(order) == list(range(n))
    early = min(R, ncl // 4)
    starts_target_only = sum(1 for cid in range(min(ncl, n)) if order[cid] >= N_d)
    # the early rows, plus first positions that lie past every paired row (tiny batches)
    assert starts_target_only == early + max(0, min(ncl, n) - (N_d + early))
    paired = [x for x in order if x < N_d]
    assert paired == list(range(N_d))
    assert [unit_at(u, N_d, R, ncl, whole_launch=False) for u in range(n)] == list(range(n))
