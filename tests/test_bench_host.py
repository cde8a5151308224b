"""Host logic of bench.py (no GPU): byte and flop accounting, the roofline
entry, the ncu-traffic lookup, the reference arm's JSON line, and the
multi-rank helpers under a two-process gloo group on CPU."""
import json
import os
import shutil
import socket

import pytest
import torch.multiprocessing as mp

import bench
import synthetic


def test_algorithmic_bytes_and_flops():
    # codes K*N/2, fp16 scales 2*G*N, int4 zero points G*N/2, A 2*M*K, Y 2*M*N
    assert bench.alg_bytes(1, 4096, 4096, 128) == 4096 * 4096 // 2 + 2 * 32 * 4096 + 32 * 4096 // 2 + 2 * 4096 + 2 * 4096
    assert bench.alg_bytes(3, 128, 16, 128) == 1024 + 32 + 8 + 768 + 96
    assert bench.flops(2, 64, 16) == 2 * 2 * 16 * 64


def test_cases_split_by_roofline_bound():
    pk = {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "measured"}
    cases = [bench.Case(*c) for c in synthetic.workload(4).cases()]
    hbm, tc = bench.split_by_bound(cases, pk)
    assert sorted(hbm + tc) == list(range(len(cases)))
    # the 70B sweep: M <= 64 is below the ridge, M >= 512 above it
    assert {cases[i].M for i in hbm} == {1, 8, 64}
    assert {cases[i].M for i in tc} == {512, 4096}
    # the headline unit follows the bound that holds most of the roofline time
    assert bench.headline_unit(synthetic.workload(4), pk) == "TFLOP/s"
    assert bench.headline_unit(synthetic.workload(1), pk) == "GB/s"


def test_group_roofline_per_bound():
    pk = {"hbm_gbs": 1000.0, "tflops": 100.0, "tflops_sustained": 80.0, "source": "measured"}
    cases = [bench.Case(*c) for c in synthetic.workload(4).cases()]
    hbm, tc = bench.split_by_bound(cases, pk)
    steps = 4
    hb = sum(bench.alg_bytes(cases[i].M, cases[i].K, cases[i].N, cases[i].group) for i in hbm)
    e = bench.group_roofline(pk, cases, hbm, secs=2e-3, steps=steps, bound="hbm", kernels={})
    # achieved = algorithmic bytes per launch / mean launch time = bytes per step / step time
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert e["achieved"] == pytest.approx(hb * steps / 2e-3 / 1e9)
    assert e["frac"] == pytest.approx(e["achieved"] / 1000.0)
    assert e["launches_per_step"] == len(hbm)
    tf = sum(bench.flops(cases[i].M, cases[i].K, cases[i].N) for i in tc)
    e = bench.group_roofline(pk, cases, tc, secs=1.0, steps=steps, bound="tensor", kernels={})
    assert e["bound"] == "tensor" and e["unit"] == "TFLOP/s"
    assert e["achieved"] == pytest.approx(tf * steps / 1.0 / 1e12)
    # tensor-bound launches are timed back to back: sustained peak, burst beside it
    assert e["peak"] == 80.0 and e["frac"] == pytest.approx(e["achieved"] / 80.0)
    assert e["frac_of_burst"] == pytest.approx(e["achieved"] / 100.0)
    roof = sum(bench.roofline_us(cases[i].M, cases[i].K, cases[i].N, cases[i].group, pk)[0]
               for i in tc) * 1e-6
    assert e["roofline_frac"] == pytest.approx(roof * steps / 1.0)


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    value = bench.profiled_traffic(1)
    assert value is None or value > 0
    # a copy of the tree whose decode kernel changed: the counters no longer apply
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    csrc = root / "bit_weight_only_g128_gb300" / "csrc"
    shutil.copytree(os.path.join(bench.ROOT, "bit_weight_only_g128_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.profiled_traffic(1) == value
    with open(csrc / "decode.cu", "a") as f:
        f.write("\n// changed\n")
    assert bench.profiled_traffic(1) is None
    assert bench.profiled_traffic(0) is None   # no summary for that workload


def test_reference_arm_line(monkeypatch, capsys):
    calls = []

    def fake_pass(wl, ncols, cache):
        calls.append(ncols)
        return 0.5, 1_000_000, 2_000_000

    monkeypatch.setattr(bench, "oracle_sample_pass", fake_pass)

    class A:
        steps, warmup = 2, 3
    wl = synthetic.workload(1)
    bench.run_reference(A, wl, None, 1, 2)       # rank 1: no work, no output
    assert calls == [] and capsys.readouterr().out == ""
    bench.run_reference(A, wl, None, 0, 2)
    line = json.loads(capsys.readouterr().out)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s"                          # the decode workload is HBM-bound
    assert line["value"] == pytest.approx(2e-3)            # 1 MB / 0.5 s in GB/s
    assert line["config"] == bench.workload_config(wl)
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert len(calls) == 1 + 3 + 2                        # probe, warm-up, timed


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist, r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank) and dist.get_backend() == "gloo"
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, 1.5 + rank)
    bench.barrier(dist)
    out[rank] = m
    dist.destroy_process_group()


def test_two_rank_max_and_barrier_under_gloo(monkeypatch):
    # CPU ranks: the helpers pick gloo when no GPU is visible
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "")
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_process_helpers_are_no_ops():
    assert bench.max_over_ranks(None, 3.0) == 3.0
    bench.barrier(None)
