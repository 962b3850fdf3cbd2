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
