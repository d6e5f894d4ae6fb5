"""Host logic of bench.py that sets the roofline numerators: the causal
(row, key) pair count of the lazy attention, the algorithmic bytes of the
streaming kernels, and the hash check that keeps a stale ncu traffic record
out of the report. No GPU needed."""
import os

import numpy as np
import torch

import bench
import synth


def test_pair_count_matches_brute_force():
    rng = np.random.default_rng(11)
    B, H, N, R, K = 3, 4, 97, 23, 19
    A = np.stack([np.sort(rng.choice(N, R, replace=False)) for _ in range(B)]).astype(np.int32)
    S = np.stack([[np.sort(rng.choice(N, K, replace=False)) for _ in range(H)] for _ in range(B)]).astype(np.int32)
    pool = np.setdiff1d(np.arange(N), A[0, :3])   # keys at exactly a row's position count (causal j <= i)
    S[0, 0] = np.sort(np.concatenate([A[0, :3], rng.choice(pool, K - 3, replace=False)]))
    want = sum(1 for b in range(B) for h in range(H) for i in A[b] for j in S[b, h] if j <= i)
    assert bench.pair_count(torch.from_numpy(A), torch.from_numpy(S)) == want


def test_pair_count_edge_sets():
    A = torch.tensor([[0, 5, 9]], dtype=torch.int32)
    assert bench.pair_count(A, torch.tensor([[[10, 11]]], dtype=torch.int32)) == 0       # every key after every row
    assert bench.pair_count(A, torch.tensor([[[0, 1, 2]]], dtype=torch.int32)) == 1 + 3 + 3
    assert bench.pair_count(A, torch.arange(10, dtype=torch.int32).view(1, 1, 10)) == 1 + 6 + 10


def test_streaming_bytes_at_32k_from_tensor_shapes():
    """Bytes rebuilt from what each kernel reads and writes at B=1, N=32768,
    H=16, d=128, R=4916, K=3277, in the first lazy loop (no earlier delta
    layer; every selected key that is also active holds a delta entry): bf16
    hidden states, int4 codes (two per byte) with one fp16 scale per 32
    elements, int32 indices and slots."""
    w = synth.WORKLOADS["32k"]
    R, K = synth.active_count(w), synth.key_count(w)
    assert (R, K) == (4916, 3277)
    got = bench.hbm_bytes(w, R, K)        # A = the first R tokens, S = the first K tokens of every head
    rows_bf16 = R * 16 * 128 * 2                       # one [R, H, d] bf16 tensor
    codes, scales = R * 16 * 64, R * 16 * 4 * 2        # [R, H, d/2] u8 and [R, H, d/32] f16
    assert got["token_scores"] == 2 * (32768 * 2048 * 2) + 32768 * 4 == 268566528
    assert got["topk_tokens"] == 32768 * 4 + R * 4
    assert got["topk_keys"] == 16 * 32768 * 4 + 16 * K * 4
    # K and V: loop-l rows and base rows read, codes and scales written; entry index and slot
    assert got["delta_append"] == 2 * (2 * rows_bf16 + codes + scales) + R * 4 * 2 == 91909536
    sel_bf16 = 16 * K * 128 * 2                        # one [H, K, d] bf16 tensor
    entry = 64 + 4 * 2                                 # one (token, head) delta entry: codes and scales
    # K and V: base rows of the selected keys and the entries of the K selected keys
    # (all active in this layer) read; key list read
    assert got["reconstruct_keys"] == 2 * (sel_bf16 + 16 * K * entry) + 16 * K * 4
    assert got["reconstruct_keys_materialised"] == got["reconstruct_keys"] + 4 * sel_bf16


def test_loop_bytes_count_earlier_entries_from_the_sets():
    """In a later lazy loop the append also reads the earlier delta entries of
    its active tokens, and the reconstruction the entries of its selected keys
    in every layer up to this loop's: counted from the set intersections."""
    w = synth.WORKLOADS["tiny"]       # B1 N1024 H4 d64, loops 2..4 lazy
    R, K = 6, 3
    act = {2: torch.tensor([[1, 3, 5, 7, 9, 11]], dtype=torch.int32),
           3: torch.tensor([[3, 4, 5, 6, 7, 8]], dtype=torch.int32)}
    keys = {2: torch.zeros(1, 4, K, dtype=torch.int32),
            3: torch.tensor([[[3, 5, 100]] * 4], dtype=torch.int32)}
    b3 = bench.loop_bytes(w, R, K, act, keys, 3)
    b2 = bench.loop_bytes(w, R, K, act, keys, 2)
    E = 4 * (32 + 4)                  # one token's entry per tensor: 4 heads x (d/2 + 2 d/32)
    assert b3["delta_append"] - b2["delta_append"] == 2 * 3 * E         # tokens 3, 5, 7 hold a loop-2 entry
    e_head = 32 + 4
    # loop 3's keys {3, 5, 100}: 3 and 5 hold entries in layers 2 and 3, in all 4 heads
    assert b3["reconstruct_keys"] == 2 * (4 * K * 64 * 2 + (2 * 4 + 2 * 4) * e_head) + 4 * K * 4


def test_recorded_traffic_needs_the_captured_source(tmp_path, monkeypatch):
    csrc = tmp_path / "lazy_sparse_attention_token_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    hdr = csrc / "h.cuh"
    hdr2 = csrc / "deep.h"
    hdr2.write_bytes(b"#define X 1\n")
    hdr.write_bytes(b'#include "deep.h"\n__device__ int f();\n')
    src.write_bytes(b'#include "h.cuh"\n#include <cuda.h>\n__global__ void k() {}\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_digest("k.cu")
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# kernel workload bytes file hash\n"
        f"k 32k 12345 k.cu {h}\n"
        f"k 8k 777 k.cu {h}\n"
        "gone 32k 1 missing.cu 0000000000000000\n")
    assert bench.recorded_traffic("k", "32k") == 12345
    assert bench.recorded_traffic("k", "8k") == 777
    assert bench.recorded_traffic("k", "deep") is None          # no capture of this workload
    assert bench.recorded_traffic("gone", "32k") is None        # source file not there
    hdr2.write_bytes(b"#define X 2\n")                          # a header two levels down changed
    assert bench.recorded_traffic("k", "32k") is None
    hdr2.write_bytes(b"#define X 1\n")
    assert bench.recorded_traffic("k", "32k") == 12345
    src.write_bytes(b'#include "h.cuh"\n#include <cuda.h>\n__global__ void k() { }\n')   # kernel changed
    assert bench.recorded_traffic("k", "32k") is None


def test_committed_traffic_record_names_existing_sources():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "profiles", "traffic.txt")) as f:
        lines = f.readlines()
    for line in lines:
        if line.startswith("#") or not line.strip():
            continue
        kernel, workload, nbytes, fname, h = line.split()
        assert int(nbytes) > 0 and len(h) == 16
        assert os.path.exists(os.path.join(root, "lazy_sparse_attention_token_b300", "csrc", fname)), fname


FAKE_SMI = r'''#!/usr/bin/env python3
# Stand-in for nvidia-smi --query-gpu ... -lms 50: 1000 MHz, no throttle reason,
# except between 0.35 s and 1.1 s after start: 2032 MHz with sw_power_cap.
import datetime, sys, time
t_start = time.time()
stamps = "{stamps}"
while True:
    t = time.time() - t_start
    hot = 0.35 <= t < 1.1
    ts = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3] if stamps == "ok" else "N/A"
    print(", ".join([ts, "0", "2032" if hot else "1000", "2032", "480.5" if hot else "90.0",
                     "0x4" if hot else "0x0", "Not Active", "Not Active", "Not Active",
                     "Active" if hot else "Not Active"]), flush=True)
    time.sleep(0.05)
'''


def _fake_smi(tmp_path, monkeypatch, stamps):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE_SMI.replace("{stamps}", stamps))
    exe.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")


def _sample(window_after_start=0.2, window_len=0.4):
    import time
    cs = bench.ClockSampler(0)
    cs.start()                       # returns 0.3 s after the sampler starts
    time.sleep(window_after_start)
    cs.mark_start()
    time.sleep(window_len)
    cs.mark_end()
    out = cs.stop()
    assert cs.proc.poll() is not None    # the sampler process has ended
    return out


def test_clock_sampler_keeps_only_the_timed_window(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch, "ok")
    out = _sample()
    assert out["window"] == "timed region"
    assert out["sm_mhz"] == 2032.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 480.5
    assert 4 <= out["samples"] <= 14     # about 0.4 s + slack at 50 ms, not the whole run


def test_clock_sampler_without_timestamps_uses_every_sample(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch, "none")
    out = _sample()
    assert out["window"].startswith("whole sampler run")
    assert out["samples"] >= 12          # the idle samples before and after are included
    assert out["reasons"] == ["sw_power_cap"]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) prints
    exactly one JSON line with the keys the benchmark contract names."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                        "--warmup", "3", "--ref-budget", "1"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["n_gpus"] == 1 and j["steps"] == 1 and j["warmup"] == 3 and j["higher_is_better"] is True
    assert j["metric"] and j["config"]["workload"].startswith("tiny") and j["data"] == "synthetic"
    # the same config object as the CUDA arm's line for this workload
    import bench
    import synth
    w = synth.WORKLOADS["tiny"]
    assert j["config"] == bench.bench_config(w, synth.active_count(w), synth.key_count(w), 1)
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == j["value"]
    # measured, not scaled: the line's time is the steps it ran
    assert abs(j["value"] * j["ms_per_step"] / 1e3 - 1024) < 1e-6 * 1024
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_leg_on_host_state():
    """The bench's cpu_baseline leg, run on the host from an oracle loop-1
    state (in place of the GPU's): the all-core and one-core figures, the CPU
    model, and the oracle's thread count restored afterwards."""
    import numpy as np
    import oracle
    w = synth.WORKLOADS["tiny"]
    R, K = synth.active_count(w), synth.key_count(w)
    inp = bench._oracle_inputs(w, w.H, "cpu")
    bench._oracle_loop1(w, inp, w.H)
    state = (torch.from_numpy(inp["qh1"].view(np.int16)).view(torch.bfloat16), torch.from_numpy(inp["o1"]),
             torch.from_numpy(inp["z1"]), torch.from_numpy(inp["c1"]))
    n0 = oracle.get_threads()
    out = bench.cpu_baseline(w, R, K, state, budget_s=0.4, device="cpu")
    assert oracle.get_threads() == n0
    assert out["kind"] == "oracle" and out["unit"] == "tokens/s" and out["value"] > 0 and out["cores"] >= 1
    # the figure is one complete lazy step, timed as it is
    assert out["sample"].startswith("one complete lazy step of the tiny workload")
    assert abs(out["value"] - w.B * w.N / out["seconds"]) <= 1e-6 * out["value"]
    st = out["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["unit"] == "tokens/s", st
    assert out["sample_all_cores"]["value"] > 0
    assert out["cpu_model"] is None or isinstance(out["cpu_model"], str)


def test_cpu_baseline_falls_back_to_the_sample_when_the_full_step_is_too_long():
    import numpy as np
    w = synth.WORKLOADS["tiny"]
    R, K = synth.active_count(w), synth.key_count(w)
    inp = bench._oracle_inputs(w, w.H, "cpu")
    bench._oracle_loop1(w, inp, w.H)
    state = (torch.from_numpy(inp["qh1"].view(np.int16)).view(torch.bfloat16), torch.from_numpy(inp["o1"]),
             torch.from_numpy(inp["z1"]), torch.from_numpy(inp["c1"]))
    out = bench.cpu_baseline(w, R, K, state, budget_s=0.4, device="cpu", full_limit_s=0.0)
    assert "not run" in out["sample"] and out["value"] == out["sample_all_cores"]["value"]
