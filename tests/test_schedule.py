"""The host ring-step scheduler against the causal rule written out on natural
token positions (brute force over every (query, key) pair)."""
import itertools

import numpy as np
import pytest

import blockwise_exact_attention_ring_gb300 as ra
import oracle


def _brute_pairs(layout, causal, N, L):
    """pairs[i, s]: visible (query, key) pairs rank i meets at ring step s,
    counted from natural positions (t of query, u of key)."""
    S = N * L
    if layout == "striped":
        order = oracle.stripe_order(S, N)          # striped row -> natural token
    else:
        order = np.arange(S)
    pos = order.reshape(N, L)                        # pos[rank, local] = natural token
    out = np.zeros((N, N), dtype=np.int64)
    for i in range(N):
        for s in range(N):
            j = (i - s) % N                          # block that reached rank i at step s
            t = pos[i][:, None]
            u = pos[j][None, :]
            out[i, s] = int((u <= t).sum()) if causal else L * L
    return out


@pytest.mark.parametrize("layout,causal,N,L", list(itertools.product(
    ["contiguous", "striped"], [False, True], [1, 2, 3, 4, 8], [1, 5, 8, 130])))
def test_pairs_per_rank_and_step_match_brute_force(layout, causal, N, L):
    total, pairs, tiles = ra.schedule_stats(layout, causal, N, L)
    assert np.array_equal(pairs, _brute_pairs(layout, causal, N, L))
    S = N * L
    assert total == (S * (S + 1) // 2 if causal else S * S)
    ntiles = -(-L // 128)
    # no visible pair is ever left out of the launched tiles
    assert np.all(tiles * 128 * 128 >= pairs)
    assert np.all(tiles <= ntiles * ntiles)


@pytest.mark.parametrize("S,expect", [(32768, 536887296), (262144, 34359869440),
                                      (1048576, 549756338176)])
def test_causal_pair_totals_at_workload_sizes(S, expect):
    # S(S+1)/2 for the 32K, 256K and 1M causal workloads
    assert S * (S + 1) // 2 == expect
    for layout, N in (("contiguous", 4), ("striped", 8)):
        if S // N > 40000:
            continue  # the per-row loop is O(N^2 L); the closed form above covers it
        total, _, _ = ra.schedule_stats(layout, True, N, S // N)
        assert total == expect


def test_striping_balances_causal_work():
    """Critical path sum_s max_i work(i, s): striping cuts it toward the mean;
    contiguous causal rank i idles for the steps s > i."""
    N, L = 8, 1024
    _, pc, _ = ra.schedule_stats("contiguous", True, N, L)
    _, ps, _ = ra.schedule_stats("striped", True, N, L)
    assert pc.sum() == ps.sum()
    assert np.count_nonzero(pc == 0) == N * (N - 1) // 2      # skipped block pairs
    assert np.count_nonzero(ps == 0) == 0                     # striped skips none
    crit_c = pc.max(axis=0).sum()   # L^2/2 + (N - 1) L^2
    crit_s = ps.max(axis=0).sum()   # N L (L + 1) / 2
    assert abs(crit_c / crit_s - (N - 0.5) / (N / 2)) < 0.01


def _brute_units(B, H, Hkv, S, N, layout, causal, steps):
    """Every (query head, query tile, rank) the kernel must cover, with the key
    tiles its ring steps visit, computed from the masks on natural positions."""
    L = S // N
    ntiles = -(-L // 128)
    order = oracle.stripe_order(S, N) if layout == "striped" else np.arange(S)
    pos = order.reshape(N, L)
    ss = range(N) if steps is None else [steps]
    need = {}
    for i in range(N):
        for ta in range(ntiles):
            t = pos[i][ta * 128:(ta + 1) * 128]
            tiles = 0
            for s in ss:
                j = (i - s) % N
                for tb in range(ntiles):
                    u = pos[j][tb * 128:(tb + 1) * 128]
                    if not causal or (u[None, :] <= t[:, None]).any():
                        tiles += 1
            for bh in range(B * H):
                need[(bh, ta, i)] = tiles
    return need


@pytest.mark.parametrize("B,H,Hkv,S,N", [(1, 4, 2, 1024, 4), (2, 3, 1, 1536, 3),
                                         (1, 2, 2, 640, 5), (1, 8, 2, 256, 2)])
@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("steps", [None, 0, 1])
def test_kernel_units_cover_every_tile_once_heaviest_first(B, H, Hkv, S, N, layout, causal, steps):
    units = ra.schedule_units(B, H, Hkv, S, N, layout, causal, steps)
    need = _brute_units(B, H, Hkv, S, N, layout, causal, steps)
    seen = {}
    for bh0, ta0, bh1, ta1, rank, cost, valid1, _ in units:
        for bh, ta, ok in ((bh0, ta0, True), (bh1, ta1, bool(valid1))):
            if not ok:
                continue
            key = (int(bh), int(ta), int(rank))
            assert key not in seen, "tile scheduled twice"
            seen[key] = int(cost)
            # both tiles of a unit read the same kv head
        g = H // Hkv
        assert (bh0 % H) // g == (bh1 % H) // g and bh0 // H == bh1 // H
    # a tile pair visits the union of its tiles' key tiles: cost >= each tile's need
    active = {k: v for k, v in need.items() if v > 0}
    assert set(seen) == set(active)
    for k, c in seen.items():
        assert c >= active[k]
    _check_order(units, H, Hkv, B * Hkv * S >= (1 << 19))


def _check_order(units, H, Hkv, kv_outer):
    costs = units[:, 5]
    assert np.all(costs > 0)
    if not kv_outer:
        assert np.all(np.diff(costs) <= 0), "not heaviest first"
        return
    # kv head outermost (the CTAs in flight share one head's K and V), and
    # heaviest first within each kv head
    g = H // Hkv
    kvh = (units[:, 0] // H) * Hkv + (units[:, 0] % H) // g
    assert np.all(np.diff(kvh) >= 0), "kv heads interleaved"
    for h in np.unique(kvh):
        c = costs[kvh == h]
        assert np.all(np.diff(c) <= 0), "not heaviest first within a kv head"


@pytest.mark.parametrize("layout,causal", [("contiguous", True), ("striped", True),
                                           ("contiguous", False)])
def test_large_problem_units_grouped_by_kv_head(layout, causal):
    """256K tokens x 8 kv heads: every tile pair listed once, kv head outermost."""
    B, H, Hkv, S, N = 1, 32, 8, 262144, 8
    units = ra.schedule_units(B, H, Hkv, S, N, layout, causal)
    L, ntiles = S // N, S // N // 128
    assert len(units) == (B * H // 2) * N * ntiles
    keys = set(map(tuple, units[:, [0, 1, 4]].tolist()))
    assert len(keys) == len(units)
    _check_order(units, H, Hkv, True)
