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
    nbytes = bench.algorithmic_bytes(c2, lens)
    tf32 = 2000.0 * 1.1 / 2.25
    # Only the method's work counts: 4*D FLOP per (row, key), not the three
    # tf32 MMAs of the emulation.  At these sizes HBM binds.
    assert flops / (tf32 * 1e12) < nbytes / 7000e9
    r = bench.roofline_for(c2, lens, 0.05, peaks, 152)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 7000.0
    assert abs(r["achieved"] - nbytes / 0.05e-3 / 1e9) < 1e-2
    assert abs(r["tensor_issue_frac"] - 3 * flops / 0.05e-3 / 1e12 / tf32) < 1e-4
    # A long fp32 problem on the same kernel is bound by the tf32 pipe.
    long = synthetic.small(dtype="f32", D=64, B=1, H=8, Lq=8192, Lk=8192, mask=0)
    r2 = bench.roofline_for(long, None, 1.0, peaks, 152)
    assert r2["bound"] == "tensor" and abs(r2["peak"] - tf32) < 0.1
    assert abs(r2["achieved"] - bench.mask_aware_flops(long, None) / 1e-3 / 1e12) < 1e-3


def test_headline_is_the_largest_config():
    assert bench.DEFAULT_WORKLOAD == "c5_long_causal_bf16"


def test_even_row_sample_accounts_exact_flops():
    for name in ("c1_causal_f32", "c2_padding_f32", "c4_prenorm_bf16"):
        w = synthetic.WORKLOADS[name]
        lens = None if w.len_range is None else list(range(w.len_range[0], w.len_range[0] + w.B))
        rows, f = bench.sample_rows_even(w, lens, 1.0)   # tiny target: stride covers all rows
        total = bench.mask_aware_flops(w, lens)
        rows1, f1 = bench.sample_rows_even(w, lens, total * 10)   # stride 1: every row
        assert len(rows1) == w.B * w.H * w.Lq and abs(f1 - total) <= 1e-9 * total
        rows4, f4 = bench.sample_rows_even(w, lens, total / 4, offset=1)
        assert abs(len(rows4) - len(rows1) / 4) <= 1
        assert 0.2 * total < f4 < 0.3 * total
        assert set(map(tuple, rows4)) <= set(map(tuple, rows1))


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


def test_nvtx_range_is_harmless_without_a_gpu():
    """The bench's NVTX ranges never raise, with or without a device."""
    import bench
    with bench.nvtx_range("phase"):
        x = 1
    assert x == 1


def test_forced_f32_kernel_changes_the_reported_kernel_and_roof(monkeypatch):
    """--f32-kernel 1 / 2 (profiling the CUDA-core kernels) must make the
    bench report those kernels and their FFMA roof, not the 3xTF32 one."""
    c1 = synthetic.WORKLOADS["c1_causal_f32"]
    c2 = synthetic.WORKLOADS["c2_padding_f32"]
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0, "_source": "test"}
    monkeypatch.setattr(bench, "F32_KERNEL", 1)
    assert bench.kernel_of(c2) == "mha_fwd_f32_kernel"
    assert bench.kernel_of(c1) == "mha_fwd_f32_kernel"
    assert not bench.uses_tf32x3(c2)
    r = bench.roofline_for(c2, [512] * 16, 0.1, peaks, 152)
    assert r["kernel"] == "mha_fwd_f32_kernel" and "tensor_issue_frac" not in r
    monkeypatch.setattr(bench, "F32_KERNEL", 2)
    assert bench.kernel_of(c1) == "mha_fwd_f32_small_kernel"   # Lk * D = 8192
    assert bench.kernel_of(c2) == "mha_fwd_f32_kernel"         # Lk * D = 32768
    monkeypatch.setattr(bench, "F32_KERNEL", 0)
    assert bench.kernel_of(c1) == "attn_fwd_tf32x3_kernel"
