"""Per-device ring steps on the host: the units ra_forward_block launches and
the lock-step critical-path model of the ring's load balance."""
import itertools

import numpy as np
import pytest

import blockwise_exact_attention_ring_gb300 as ra
from blockwise_exact_attention_ring_gb300 import balance


@pytest.mark.parametrize("B,H,Hkv,S,N", [(1, 4, 2, 1024, 4), (2, 3, 1, 1536, 3), (1, 2, 2, 640, 5),
                                         (1, 32, 8, 262144, 8)])
@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True),
                                           ("contiguous", False), ("striped", False)])
def test_block_units_are_one_ranks_share_of_the_step(B, H, Hkv, S, N, layout, causal):
    """ra_forward_block(rank, step) launches exactly the units of ring step
    `step` that belong to query block `rank`, in the same heaviest-first order."""
    for s in range(N):
        step_units = ra.schedule_units(B, H, Hkv, S, N, layout, causal, s)
        seen = 0
        for i in range(N):
            got = ra.block_units(B, H, Hkv, S, N, layout, causal, i, s)
            want = step_units[step_units[:, 4] == i]
            assert np.array_equal(got, want), (s, i)
            assert np.all(got[:, 4] == i)
            seen += len(got)
        assert seen == len(step_units)


def test_block_units_empty_for_masked_block():
    """Contiguous causal: query block i sees nothing of block j > i, which it
    holds at steps s > i."""
    N = 4
    for i, s in itertools.product(range(N), range(N)):
        n = len(ra.block_units(1, 2, 1, 1024, N, "contiguous", True, i, s))
        assert (n == 0) == (s > i)


def test_block_units_rejects_bad_rank_or_step():
    L = ra.lib()
    for rank, step in [(-1, 0), (4, 0), (0, -1), (0, 4)]:
        assert L.ra_schedule_block_units(1, 2, 1, 1024, 4, 0, 1, rank, step, None, 0) == -1


@pytest.mark.parametrize("N,L", [(1, 7), (2, 128), (4, 1000), (8, 32768), (32, 32768)])
def test_critical_path_closed_forms(N, L):
    """Visible pairs per (device, step), summed over the slowest device of
    each step.  Contiguous causal: step 0 is the diagonal block L(L+1)/2,
    every later step has a device with a full block L^2.  Striped causal:
    every step has a device on an inclusive diagonal block, L(L+1)/2.
    Non-causal: L^2 everywhere, no imbalance."""
    S = N * L
    total = S * (S + 1) / 2
    c = balance.model("contiguous", True, N, L)
    s = balance.model("striped", True, N, L)
    f = balance.model("striped", False, N, L)
    assert c["total"] == total and s["total"] == total
    assert c["critical_path"] == L * (L + 1) / 2 + (N - 1) * L * L
    assert s["critical_path"] == N * L * (L + 1) / 2
    assert c["ideal"] == pytest.approx(total / N)
    assert f["critical_path"] == N * L * L and f["imbalance"] == 1.0
    assert c["imbalance"] == pytest.approx(c["critical_path"] / (total / N))
    # striping never loses, and gains ~ (2N - 1) / N for large blocks
    assert s["critical_path"] <= c["critical_path"]
    if N > 1 and L >= 1000:
        assert c["critical_path"] / s["critical_path"] == pytest.approx((2 * N - 1) / N, rel=2e-3)


def test_tile_model_counts_masked_half_of_diagonal_tiles():
    """In tiles, a diagonal block of T tiles costs T(T+1)/2 launched tiles
    (the masked upper half of each diagonal tile still runs)."""
    N, L = 4, 512
    T = L // 128
    c = balance.model("contiguous", True, N, L, unit="tiles")
    assert c["step_max"][0] == T * (T + 1) / 2
    assert all(m == T * T for m in c["step_max"][1:])


def test_measured_summary_matches_model_on_model_input():
    _, pairs, _ = ra.schedule_stats("contiguous", True, 8, 256)
    assert balance.measured(pairs)["critical_path"] == balance.model("contiguous", True, 8, 256)[
        "critical_path"]
    with pytest.raises(ValueError):
        balance.summarize(np.zeros((2, 3)))


def _visible_tile_pairs(B, H, S, N, layout, causal):
    """(bh, i, ta, j, tb) for every query tile / key tile pair with a visible
    (query, key) pair, from the causal rule on natural positions."""
    import oracle
    L = S // N
    nt = -(-L // 128)
    order = oracle.stripe_order(S, N) if layout == "striped" else np.arange(S)
    pos = order.reshape(N, L)
    out = set()
    for i in range(N):
        for ta in range(nt):
            t = pos[i][ta * 128:(ta + 1) * 128]
            for j in range(N):
                for tb in range(nt):
                    u = pos[j][tb * 128:(tb + 1) * 128]
                    if not causal or (u[None, :] <= t[:, None]).any():
                        for bh in range(B * H):
                            out.add((bh, i, ta, j, tb))
    return out


@pytest.mark.parametrize("B,H,Hkv,S,N", [(1, 4, 2, 1024, 4), (2, 3, 1, 768, 3), (1, 2, 2, 640, 5),
                                         (8, 128, 64, 1024, 4)])  # 2^19 K/V rows: units grouped by kv head
@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("contiguous", False)])
def test_backward_kernels_cover_every_visible_tile_pair_once(B, H, Hkv, S, N, layout, causal):
    """Both backward kernels visit exactly the tile pairs with a visible key,
    each once; the dK/dV kernel meets query blocks in the order the key block
    travels (i = j, j + 1, ...) and the dQ kernel key blocks in the forward's
    order (j = i, i - 1, ...)."""
    want = _visible_tile_pairs(B, H, S, N, layout, causal)
    for which in (0, 1):
        pairs = ra.backward_tile_pairs(B, H, Hkv, S, N, layout, causal, which)
        got = [tuple(r) for r in pairs[:, 1:6].tolist()]
        assert len(got) == len(set(got)) == len(want), which
        assert set(got) == want, which
        for u in np.unique(pairs[:, 0]):
            rows = pairs[pairs[:, 0] == u]
            assert np.array_equal(rows[:, 6], np.arange(len(rows)))
            steps = (rows[:, 2] - rows[:, 4]) % N if which == 0 else (rows[:, 2] - rows[:, 4]) % N
            assert np.all(np.diff(steps) >= 0), (which, u)
            if which == 0:
                grp = H // Hkv
                assert len(set((rows[:, 1] // H * Hkv + rows[:, 1] % H // grp).tolist())) == 1
                assert len(set(rows[:, 4].tolist())) == 1 and len(set(rows[:, 5].tolist())) == 1
            else:
                assert len(set(rows[:, 1].tolist())) == 1 and len(set(rows[:, 3].tolist())) == 1


@pytest.mark.parametrize("B,H,Hkv,S,N", [(1, 8, 2, 1024, 4), (2, 16, 4, 768, 3), (1, 32, 8, 262144, 8),
                                         (1, 8, 1, 640, 5), (1, 32, 8, 1048576, 32)])
@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("striped", False)])
def test_cluster_pairs_share_one_key_walk(B, H, Hkv, S, N, layout, causal):
    """Kernel variant 3 deals units (2m, 2m + 1) to the two CTAs of a cluster,
    which share every key/value tile load: with four or more query heads per
    kv head (an even number of head pairs), both units of each pair have the
    same kv head, rank and query tiles, so they walk the same key tiles, and
    they differ in their query heads."""
    u = ra.schedule_units(B, H, Hkv, S, N, layout, causal)
    assert len(u) % 2 == 0
    a, b = u[0::2], u[1::2]
    grp = H // Hkv
    kv = lambda bh: (bh // H) * Hkv + (bh % H) // grp
    assert np.array_equal(kv(a[:, 0]), kv(b[:, 0]))
    assert np.array_equal(a[:, [1, 3, 4, 5, 6]], b[:, [1, 3, 4, 5, 6]])
    assert np.all(a[:, 0] != b[:, 0]) and np.all(a[:, 2] != b[:, 2])


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True), ("contiguous", False)])
def test_cluster_pairs_within_one_devices_step(layout, causal):
    """ra_forward_block restricts the unit space to one rank and one ring
    step; its units still pair up (2m, 2m + 1) on one key walk, so the
    K/V-sharing CTA pairs serve one device's step as well."""
    B, H, Hkv, S, N = 1, 8, 2, 2048, 4
    grp = H // Hkv
    kv = lambda bh: (bh // H) * Hkv + (bh % H) // grp
    for i in range(N):
        for s in range(N):
            u = ra.block_units(B, H, Hkv, S, N, layout, causal, i, s)
            assert len(u) % 2 == 0
            if len(u) == 0:
                continue
            a, b = u[0::2], u[1::2]
            assert np.array_equal(kv(a[:, 0]), kv(b[:, 0]))
            assert np.array_equal(a[:, [1, 3, 4, 5, 6]], b[:, [1, 3, 4, 5, 6]])


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_backward_units_grouped_by_kv_head_on_large_problems(layout):
    """From 2^19 key/value rows the backward kernels deal their units kv head
    by kv head (the units in flight then stream one kv group's data), as the
    forward does; below it the head index runs fastest."""
    B, H, Hkv, S, N = 8, 128, 64, 1024, 4           # B * Hkv * S = 2^19
    grp = H // Hkv
    for which in (0, 1):
        pairs = ra.backward_tile_pairs(B, H, Hkv, S, N, layout, True, which)
        units = pairs[np.unique(pairs[:, 0], return_index=True)[1]]
        kv = units[:, 1] // H * Hkv + units[:, 1] % H // grp
        assert np.all(np.diff(kv) >= 0), which      # kv head outermost, non-decreasing
    small = ra.backward_tile_pairs(1, 4, 2, 1024, 4, layout, True, 1)
    units = small[np.unique(small[:, 0], return_index=True)[1]]
    assert list(units[:4, 1]) == [0, 1, 2, 3]       # head fastest below the threshold
