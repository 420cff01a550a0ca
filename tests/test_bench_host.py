"""Host-side logic of bench.py: algorithmic work counts and the multi-rank
timing reduction (run as two gloo ranks on the CPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import mc_inputs


def test_algorithmic_flops_long_grm():
    w = mc_inputs.LONG_GRM
    f = bench.algorithmic_flops(w)
    # GRM: sum_t (s_t - 1) = C * N (N - 1) / 2 with C = L / N
    per_head = w.L * 4 * w.d ** 2 + 2 * w.d ** 2 * (w.seg_len * w.N * (w.N - 1) // 2) \
        + 2 * w.d * (w.seg_len * w.N * (w.N + 1) // 2)
    assert f["total"] == w.B * w.H * per_head
    assert abs(f["total"] / 1e12 - 1.16) < 0.01  # ~ L d^2 (N + 3) per head


def test_algorithmic_flops_modes():
    w = mc_inputs.SSC_D128
    f = bench.algorithmic_flops(w)
    s, n = bench.segment_counts(w)
    assert max(n) == w.topk and n[0] == 0
    r = bench.algorithmic_flops(w.with_(mode=mc_inputs.RESIDUAL))
    online_read = w.B * w.H * w.L * 2 * w.d ** 2  # M_t q_t per token
    assert r["readout"] == online_read and r["total"] == r["online"] == r["state"] + r["readout"]
    assert f["total"] == f["state"] + f["readout"] > r["total"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank
    mx = bench.reduce_max(ms, dist)
    val = bench.aggregate(1000, 4, mx, world)
    out[rank] = (mx, val)
    dist.barrier()
    dist.destroy_process_group()


def test_backward_flops_tensor_core_split():
    # the tensor-core backward's kernels share the stated work exactly (the gates kernel
    # recomputes forward work, outside the total)
    w = mc_inputs.LONG_GRM
    f = bench.backward_flops(w)
    tc = ("seg_state_tc", "bwd_cached_tc", "bwd_route_simt", "bwd_dkbar_tc", "bwd_G_tc", "bwd_kv_tc")
    assert sum(f[k] for k in tc) == f["total"]
    assert f["gate_tiles_tc"] == w.B * w.H * 2 * w.d * sum(t // w.seg_len for t in range(w.L))
    assert abs(f["total"] / 1e12 - 3.4019) < 1e-3
    r = bench.backward_flops(w.with_(mode=mc_inputs.RESIDUAL))
    assert r["gate_tiles_tc"] == 0 and r["bwd_route_simt"] == 0


def test_reduce_max_two_gloo_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    mx, val = out[0]
    assert mx == 15.0
    assert val == pytest.approx(1000 * 4 * 2 / 0.015)


def test_single_rank_reduce_is_identity():
    assert bench.reduce_max(3.5, None) == 3.5


def test_roofline_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """`traffic` comes from a committed ncu summary only while the kernel sources it
    was taken on are unchanged (the summary records their sha256)."""
    for rel in set(bench.KERNEL_SOURCES + bench.GEN_KERNEL_SOURCES):
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_text("kernel source " + rel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    summary = tmp_path / "profiles" / "readout_tc_long-grm.md"
    assert bench.ncu_traffic("readout_tc", "long-grm") is None  # no summary
    summary.write_text(f"# x\n\n- kernel_source_sha256: `{bench.kernel_source_hash()}`\n"
                       "- traffic_bytes_per_launch: 1698533376\n")
    assert bench.ncu_traffic("readout_tc", "long-grm") == 1698533376
    (tmp_path / bench.KERNEL_SOURCES[0]).write_text("changed")
    assert bench.ncu_traffic("readout_tc", "long-grm") is None
    assert bench.ncu_traffic("gates_tc", "long-grm") is None
    fact = tmp_path / "profiles" / "readout_fact_tc_fact-c32.md"
    fact.write_text(f"- kernel_source_sha256: `{bench.kernel_source_hash('readout_fact_tc')}`\n"
                    "- traffic_bytes_per_launch: 123\n")
    assert bench.ncu_traffic("readout_fact_tc", "fact-c32") == 123  # the state-form sources do not matter to it


def test_workload_bounds_and_kernel_bytes():
    """The long workload is bound by the tensor cores, the sweep's short-N rows, the d = 64
    workload and SSC by HBM; each kernel's algorithmic bytes add up to the step's bytes
    plus the inputs both kernels must read (k, v and u twice) and the bf16 state reads."""
    peaks = {"bf16_tflops": 1946.8, "hbm_gbs": 6775.6}
    assert bench.workload_bound(mc_inputs.LONG_GRM, peaks) == "tensor"
    assert bench.workload_bound(mc_inputs.SSC_D128, peaks) == "hbm"
    assert bench.workload_bound(mc_inputs.GRM_D64, peaks) == "hbm"
    assert [bench.workload_bound(w, peaks) for w in mc_inputs.SWEEP] == ["hbm", "hbm", "hbm", "tensor"]
    w = mc_inputs.LONG_GRM
    kb = bench.kernel_bytes(w)
    row = w.B * w.H * w.L * w.d * 2
    urow0 = w.B * w.H * w.seg_len * w.d * 2  # u of the first segment is not read
    assert kb["seg_state_tc"] + kb["readout_tc"] == bench.algorithmic_bytes(w) + 3 * row - 2 * urow0 + \
        w.B * w.H * w.N * w.d * w.d * 2
    assert bench.metric_name(w) == bench.METRIC
    assert "SSC" in bench.metric_name(mc_inputs.SSC_D128)


def test_reference_arm_reports_the_gpu_arms_config(monkeypatch):
    """Both arms print one config object for a workload: the same keys and values, including
    how the timed steps treat the L2 and the replica layout."""
    w = mc_inputs.TINY
    monkeypatch.setattr(bench, "oracle_sample", lambda w, budget_s: (1.0, 1, "stub sample", None))
    monkeypatch.setattr(bench, "dist_env", lambda: (1, 0, 0))

    class Args:
        steps, warmup = 1, 0

    line = bench.run_reference(Args, w)
    note = bench.l2_note(bench.forward_inputs_bytes(w))
    assert line["config"] == bench.forward_config(w, 1, note)
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert "fit in L2" in note
    assert "not flushed" in bench.l2_note(bench.forward_inputs_bytes(mc_inputs.LONG_GRM))
    assert set(line["config"]) >= {"workload", "B", "H", "L", "d", "seg_len", "N", "agg", "topk", "input_dtype",
                                   "l2", "parallelism"}
