"""Host logic of bench.py: FLOP and byte accounting, and the weak-scaling
combination of replica timings over a world-size-2 gloo group (CPU only)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from masked_head_attention_gb300 import synthetic


def test_mask_aware_flops():
    w = synthetic.WORKLOADS["c1_causal_f32"]
    assert bench.mask_aware_flops(w, None) == 4 * 4 * 8 * 128 * 128 * 64 / 2
    w2 = synthetic.WORKLOADS["c2_padding_f32"]
    lens = [1, 512, 600, -4] + [256] * 12
    want = 4 * 8 * 64 * 512 * (1 + 512 + 512 + 0 + 256 * 12)
    assert bench.mask_aware_flops(w2, lens) == want
    assert bench.nominal_flops(w2) == 4 * 16 * 8 * 512 * 512 * 64


def test_algorithmic_bytes():
    w = synthetic.WORKLOADS["c3_causal_bf16"]
    assert bench.algorithmic_bytes(w, None) == 4 * 32 * 2048 * 128 * 2


def test_backward_accounting():
    w = synthetic.WORKLOADS["b2_padding_f32_bwd"]
    lens = [100, 512] + [0] * 14
    assert bench.mask_aware_flops(w, lens) == 10 * 8 * 64 * 512 * 612
    w3 = synthetic.WORKLOADS["b3_causal_f32_bwd"]
    assert bench.mask_aware_flops(w3, None) == 10 * 2 * 16 * 1024 * 1024 * 128 / 2
    rows_q = 16 * 8 * 512
    want = 4 * rows_q * 64 * 4 + 4 * rows_q + 2 * 612 * 8 * 64 * 4 + 2 * 16 * 8 * 512 * 64 * 4
    assert bench.algorithmic_bytes(w, lens) == want
    assert bench.kernel_of(w) == "mha_bwd_f32_kernel"
    small = synthetic.small(kind="mha_bwd", Lq=64, Lk=64)
    assert bench.kernel_of(small) == "mha_bwd_f32_kernel"
    b5 = synthetic.WORKLOADS["b5_causal_bf16_bwd"]
    assert bench.kernel_of(b5) == "attn_bwd_bf16_kernel"
    r = bench.roofline_for(b5, None, 1.0, {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0,
                                           "_source": "test"}, 152)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0   # bf16 backward: tensor cores


def test_kernel_choice_and_tf32_roofline():
    c2 = synthetic.WORKLOADS["c2_padding_f32"]
    assert bench.kernel_of(c2) == "attn_fwd_tf32x3_kernel"
    d128 = synthetic.small(dtype="f32", D=128, Lq=512, Lk=512)
    assert bench.kernel_of(d128) == "mha_fwd_f32_kernel"
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0, "_source": "test"}
    lens = [512] * 16
    flops = bench.mask_aware_flops(c2, lens)
    r = bench.roofline_for(c2, lens, 0.05, peaks, 152)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["peak"] - 2000.0 * 1.1 / 2.25) < 0.1
    assert abs(r["achieved"] - 3 * flops / 0.05e-3 / 1e12) < 1e-3


def test_fp32_alu_peak():
    assert abs(bench.fp32_alu_peak_tflops(152, 2070.0) - 80.54) < 0.01


def test_combine_single_rank():
    ms, tf = bench.combine_ranks(10.0, 1e12, 10, 1)
    assert ms == 1.0 and abs(tf - 1000.0) < 1e-9


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        def rmax(x):
            t = torch.tensor([float(x)], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())
        # rank r ran 20 steps in (100 + 50 r) ms, each step 2e9 FLOP
        ms, tf = bench.combine_ranks(100.0 + 50.0 * rank, 2e9, 20, world, rmax)
        q.put((rank, ms, tf))
    finally:
        dist.destroy_process_group()


def test_combine_ranks_gloo_world2():
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
    for rank, ms, tf in res:
        assert ms == pytest.approx(150.0 / 20)           # slowest rank
        assert tf == pytest.approx(2 * 2e9 / (7.5e-3) / 1e12)
