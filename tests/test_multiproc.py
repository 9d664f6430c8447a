"""The benchmark's multi-rank path on CPU: world_size 2 over gloo.

Each GPU runs an independent replica of the layer (the path has no exchange
step), so the only cross-rank logic is the barrier, the maximum of the timed
region over ranks and the whole-job value; the reference arm runs on rank 0
only.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(1.5 + rank, device="cpu")
        out.put((rank, t, bench.whole_job_value(4096, 10, world, t)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert res[0][2] == pytest.approx(4096 * 10 * 2 / 2.5)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25, device="cpu") == 3.25
    assert bench.whole_job_value(4096, 5, 1, 2.0) == pytest.approx(10240.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 0

    from combine_router_gemm_gb300 import inputs
    assert bench.run_reference(Args(), inputs.CONFIGS["tiny_fp32"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line_tiny():
    """`bench.py --impl reference` times the CPU oracle and prints one JSON line
    with the contract's keys (tiny fp32 workload, CPU only)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny_fp32",
                        "--steps", "2", "--warmup", "1"], cwd=root, capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    assert j["steps"] == 2 and j["higher_is_better"] is True


@pytest.mark.parametrize("sigmoid", [False, True])
def test_eager_comparator_computes_the_layer(oracle, sigmoid):
    """The bench's PyTorch comparator computes the same layer as the oracle
    (run here on CPU tensors; it rounds g and u to bf16 where the oracle
    keeps them in fp32, hence the looser tolerance)."""
    import numpy as np
    from combine_router_gemm_gb300 import inputs
    if sigmoid:
        cfg = inputs.MoEConfig("t", T=48, d=64, E=16, k=4, I=32, score_fn="sigmoid", n_group=4,
                               topk_group=2, routed_scale=2.5, shared_I=32, bias="normal")
    else:
        cfg = inputs.MoEConfig("m", T=48, d=64, E=8, k=2, I=48)
    inp = inputs.make_inputs(cfg, seed=0, device="cpu")
    out = bench.eager_layer(cfg, inp).numpy().astype(np.float64)
    n = inputs.to_numpy
    opt = lambda key: None if inp[key] is None else n(inp[key])
    _, _, ref = oracle.moe_tokens(n(inp["x"]), E=cfg.E, k=cfg.k, w13=n(inp["w13"]), w2=n(inp["w2"]),
                                  w_router=n(inp["w_router"]), bias=opt("bias"),
                                  n_group=cfg.n_group, topk_group=cfg.topk_group,
                                  score_fn=oracle.SIGMOID if sigmoid else oracle.SOFTMAX,
                                  routed_scale=cfg.routed_scale, w13_sh=opt("w13_sh"),
                                  w2_sh=opt("w2_sh"), round_h=True)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 1e-2
