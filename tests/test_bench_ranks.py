"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each an
independent replica, combine into whole-job throughput with the slowest
rank's time (max over ranks) and a barrier."""

import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, lr = bench.dist_env()
    dist = bench.init_dist(w)
    bench.barrier(dist)
    my_seconds = 0.5 + rank                 # rank 1 is the slow one
    worst = bench.reduce_max(dist, my_seconds)
    value = bench.aggregate(100.0, worst, w)
    bench.barrier(dist)
    q.put((r, w, lr, worst, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, lr, worst, value) in enumerate(res):
        assert (r, w, lr) == (rank, world, rank)
        assert worst == 1.5                 # max over ranks
        assert value == 100.0 * 2 / 1.5     # all ranks' units / slowest time


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1) is None
    assert bench.reduce_max(None, 3.0) == 3.0
    assert bench.aggregate(10.0, 2.0, 1) == 5.0


def test_secondary_line_is_compact_and_ends_with_the_targets():
    """The driver keeps the tail of the JSON line: the two target workloads come last
    in `secondary`, each workload reduced to a few numbers."""
    full = {k: {"workload": "w" * 200, "note": "n" * 200, "lengths": list(range(50)), "us_per_step": 1.0,
                "GBps": 2.0, "frac_of_hbm": 0.5, "frac_of_8TBps": 0.4, "TFLOPs": 3.0, "us_per_step_graph": 4.0}
            for k in ("layer_c4", "mlp_fwd_c1", "decode_c3")}
    comp = {k: bench.compact_secondary(k, v) for k, v in full.items()}
    assert list(comp)[-2:] == ["mlp_fwd_c1", "decode_c3"]
    assert comp["decode_c3"] == {"us_per_step": 1.0, "GBps": 2.0, "frac_of_hbm": 0.5, "frac_of_8TBps": 0.4}
    assert comp["mlp_fwd_c1"] == {"us_per_step": 1.0, "TFLOPs": 3.0, "us_per_step_graph": 4.0}
    assert all("workload" not in v and "lengths" not in v for v in comp.values())


class _RoundedOracleGpu:
    """Stands in for the GPU leg on CPU: the oracle's own outputs rounded to bf16, so the
    parity figures must come out small but not zero."""

    def run(self, inp_cpu, M, h, F, t, act_name, backward):
        import torch
        import oracle as O
        from megatron_tensor_transformer_shard_gb300 import inputs as I
        r = {k: O.bf16_to_f64(I.bits(v)).reshape(tuple(v.shape)) for k, v in inp_cpu.items() if v is not None}
        f = O.mlp_forward_sharded(r["X"], r["W_up"], r.get("b_up"), r["W_down"], r.get("b_down"), act_name, t)
        out = {"Y": torch.from_numpy(f["Y"]).to(torch.bfloat16)}
        if backward:
            b = O.mlp_backward_sharded(r["dY"], r["X"], r["W_up"], r["W_down"], f, act_name, t)
            out["dX"] = torch.from_numpy(b["dX"]).to(torch.bfloat16)
        return out


def test_cpu_baseline_reports_parity_of_the_benchmarked_configs():
    cb, parity = bench.cpu_baseline(budget_s=0.01, gpu=_RoundedOracleGpu(), per_config=False)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert parity["c2"]["rows"] == 128 and parity["c1"]["rows"] == 128
    for v in (parity["c2"]["Y"], parity["c2"]["dX"], parity["c1"]["Y"]):
        assert 0 < v < 2 ** -7            # bf16 rounding of the oracle's own values
    assert parity["bound"] == 1e-2


def test_single_thread_oracle_probe_runs_in_its_own_interpreter():
    r = bench._probe_subprocess("c1", 0, 1)
    assert r["seconds"] > 0 and r["sample"].startswith("the whole forward")
