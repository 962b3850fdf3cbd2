"""The communication model of the 4D grid (CPU tool).  The pages give its
assumptions but not its equations, so these are checks of the ring-cost
algebra and of the model's structure, not parity with the pages."""
import pytest

from pmm_fc_layer_gb300 import perf_model as pm

M = pm.Machine(gpus_per_node=8, inter_node_gbs=50.0, intra_node_gbs={2: 400.0, 4: 380.0, 8: 350.0})
GPT = [(6144, 18432), (6144, 6144), (6144, 24576), (24576, 6144)]


def test_ring_costs():
    assert pm.ring_time("all_reduce", 1e9, 1, 100.0) == 0.0
    for p in (2, 4, 8, 64):
        rs = pm.ring_time("reduce_scatter", 1e9, p, 100.0)
        assert rs == pytest.approx((p - 1) / p * 1e9 / 100e9)
        assert pm.ring_time("all_gather", 1e9, p, 100.0) == pytest.approx(rs)
        assert pm.ring_time("all_reduce", 1e9, p, 100.0) == pytest.approx(2 * rs)
        assert pm.ring_time("all_reduce", 2e9, p, 100.0) == pytest.approx(4 * rs)
        assert pm.ring_time("all_reduce", 1e9, p, 200.0) == pytest.approx(rs)


def test_group_placement():
    g = (2, 2, 2, 2)                       # 16 GPUs on two nodes of 8
    assert pm.axis_stride(g, "x") == 1 and pm.axis_stride(g, "data") == 8
    assert pm.group_bandwidth(g, "x", M) == 400.0     # ranks 0,1: one node
    assert pm.group_bandwidth(g, "z", M) == 400.0     # ranks 0,4: one node
    assert pm.group_bandwidth(g, "data", M) == 50.0   # ranks 0,8: two nodes
    assert pm.group_bandwidth((1, 1, 1, 16), "z", M) == 50.0


def test_single_gpu_and_pure_data_parallel():
    assert sum(pm.layer_comm(8192, 6144, 6144, (1, 1, 1, 1), M).values()) == 0.0
    c = pm.layer_comm(8192, 6144, 6144, (16, 1, 1, 1), M)
    assert c["data_allreduce_dw"] == pytest.approx(
        pm.ring_time("all_reduce", 2 * 6144 * 6144, 16, 50.0))
    assert sum(v for k, v in c.items() if k != "data_allreduce_dw") == 0.0


def test_3d_collectives_sizes():
    T, K, N, g = 8192, 6144, 24576, (1, 2, 2, 2)
    c = pm.layer_comm(T, K, N, g, M)
    w_blk = 2 * (K / 2) * (N / 2)
    assert c["fwd_allgather_w_z"] == pytest.approx(pm.ring_time("all_gather", w_blk, 2, 400.0))
    assert c["fwd_allreduce_y_x"] == pytest.approx(
        pm.ring_time("all_reduce", 2 * (T / 2) * (N / 2), 2, 400.0))
    assert c["dgrad_allreduce_dx_y"] == pytest.approx(
        pm.ring_time("all_reduce", 2 * (T / 2) * (K / 2), 2, 400.0))
    assert c["wgrad_reducescatter_dw_z"] == pytest.approx(pm.ring_time("reduce_scatter", w_blk, 2, 400.0))


def test_rank_configs_enumerates_and_orders():
    ranked = pm.rank_configs(GPT, 32768, 16, M)
    grids = [g for _, g in ranked]
    assert len(grids) == len(set(grids)) == len(list(pm.factorizations(16)))
    assert all(a <= b for (a, _), (b, _) in zip(ranked, ranked[1:]))
    for g in grids:
        assert g[0] * g[1] * g[2] * g[3] == 16
    # compute per GPU is the same for every grid of the same GPU count
    comp = {round(pm.step_time(GPT, 32768, g, M)["compute"], 12) for g in grids}
    assert len(comp) == 1
    # with a slow network the fastest grid keeps its 3D groups inside a node
    best = ranked[0][1]
    assert best[1] * best[2] * best[3] <= 8


def _ring(p, chunks, mode):
    """A literal ring on p ranks, each holding p chunks (numpy arrays).
    reduce_scatter: after p-1 steps rank r holds the sum of chunk (r+1) % p.
    all_gather: rank r starts with its own chunk (r+1) % p and ends with all.
    Returns (per-rank data, bytes each rank sent)."""
    import numpy as np
    data = [[None if c is None else np.array(c, dtype=np.float64) for c in row] for row in chunks]
    sent = [0] * p
    for step in range(p - 1):
        msgs = []
        for r in range(p):
            if mode == "reduce_scatter":
                idx = (r - step) % p
            else:
                idx = (r + 1 - step) % p
            msgs.append(((r + 1) % p, idx, data[r][idx].copy()))
            sent[r] += data[r][idx].nbytes
        for dst, idx, buf in msgs:
            data[dst][idx] = data[dst][idx] + buf if mode == "reduce_scatter" else buf
    return data, sent


@pytest.mark.parametrize("p", [2, 3, 4, 8])
def test_ring_cost_matches_a_simulated_ring(p):
    """Assumption 1 pinned by simulation, not by the formula: a ring
    reduce-scatter and all-gather of S bytes each send (p-1)/p * S bytes per
    rank, and the all-reduce (one then the other) 2 (p-1)/p * S; the
    simulated ring also yields the right sums."""
    import numpy as np
    rng = np.random.default_rng(p)
    n = 6                                        # elements per chunk
    x = rng.integers(-9, 9, size=(p, p, n)).astype(np.float64)   # rank, chunk, element
    S = p * n * 8                                # bytes of one rank's tensor
    rs, sent_rs = _ring(p, [[x[r, c] for c in range(p)] for r in range(p)], "reduce_scatter")
    total = x.sum(axis=0)
    for r in range(p):
        assert np.array_equal(rs[r][(r + 1) % p], total[(r + 1) % p])
    ag_in = [[rs[r][c] if c == (r + 1) % p else None for c in range(p)] for r in range(p)]
    ag, sent_ag = _ring(p, ag_in, "all_gather")
    for r in range(p):
        assert np.array_equal(np.stack(ag[r]), total)          # all-reduce done
    gbs = 1.0                                                  # 1 GB/s: seconds = bytes / 1e9
    assert max(sent_rs) / 1e9 == pytest.approx(pm.ring_time("reduce_scatter", S, p, gbs))
    assert max(sent_ag) / 1e9 == pytest.approx(pm.ring_time("all_gather", S, p, gbs))
    assert (max(sent_rs) + max(sent_ag)) / 1e9 == pytest.approx(
        pm.ring_time("all_reduce", S, p, gbs))


@pytest.mark.parametrize("grid", [(2, 2, 2, 2), (1, 2, 4, 2), (4, 1, 1, 4), (1, 8, 1, 2),
                                  (2, 1, 8, 1), (1, 1, 1, 16), (1, 3, 2, 1), (2, 3, 1, 1),
                                  (1, 1, 3, 4), (3, 2, 2, 1), (1, 5, 1, 3), (1, 6, 2, 2)])
def test_group_placement_by_enumeration(grid):
    """Ranks numbered x fastest, then y, z, data; a group along an axis is the
    ranks that share every other coordinate.  Enumerate the groups and check
    that the model's choice of intra- or inter-node bandwidth is intra
    exactly when every group lies within one node of 8."""
    gd, gx, gy, gz = grid
    ext = {"x": gx, "y": gy, "z": gz, "data": gd}
    coords = {}
    r = 0
    for d in range(gd):
        for z in range(gz):
            for y in range(gy):
                for x in range(gx):
                    coords[r] = {"x": x, "y": y, "z": z, "data": d}
                    r += 1
    for axis in ("x", "y", "z", "data"):
        groups = {}
        for rank, c in coords.items():
            key = tuple(v for a, v in sorted(c.items()) if a != axis)
            groups.setdefault(key, []).append(rank)
        assert all(len(g) == ext[axis] for g in groups.values())
        one_node = all(len({rank // M.gpus_per_node for rank in g}) == 1
                       for g in groups.values())
        assert pm.groups_within_nodes(grid, axis, M.gpus_per_node) == one_node
        if ext[axis] > 1:                        # a one-rank group moves nothing
            bw = pm.group_bandwidth(grid, axis, M)
            assert bw == (M.intra(ext[axis]) if one_node else M.inter_node_gbs)
