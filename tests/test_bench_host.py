"""Host-side logic of bench.py, on CPU: FLOP accounting, clock parsing, the
multi-rank (gloo, world size 2) max-over-ranks timing and the reference arm."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_flop_conventions():
    assert bench.formula_fwd_flops(1, 32, 16384, 128, True) == pytest.approx(2.199e12, rel=1e-3)
    assert bench.formula_fwd_flops(16, 16, 512, 64, False) == pytest.approx(17.18e9, rel=1e-3)


def test_visited_tile_pairs():
    assert bench.visited_tile_pairs(512, True, None, None, 1, 1) == 10
    assert bench.visited_tile_pairs(512, False, None, None, 2, 3) == 6 * 16
    # key padding: lengths 129 and 512 -> 2 and 4 key tiles for each of 4 query tiles
    assert bench.visited_tile_pairs(512, False, np.array([129, 512]), None, 2, 1) == 4 * 2 + 4 * 4
    bm = np.eye(4, dtype=np.uint8)
    assert bench.visited_tile_pairs(512, False, None, bm, 1, 2) == 8
    assert bench.visited_tile_pairs(300, True, None, None, 1, 1) == 6  # T = 3


def test_clock_parsing():
    lines = ["0, 1965, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 1980, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 1950, 2070, 990.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    s = bench.parse_clock_lines(lines)
    assert s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_lines([])["sm_mhz"] is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.reduce_max_over_ranks(1.0 + rank, dist)
    value = bench.aggregate_line(per_rank_flops=1e12, world=world, max_ms_step=slowest, steps=10)
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_two():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # both ranks see the slower rank's 2 ms, and the job throughput counts both ranks' work
    assert res[0] == res[1] == (2.0, pytest.approx(2e12 / 2e-3 / 1e12))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_warmup_floor():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "1"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0


def test_kernel_digest_ignores_comments_only():
    a = "int f(int x) {  // scale\n  return 2 * x; /* twice */\n}\n"
    b = "// a new comment\nint f(int x) {\n\n  return 2 * x;\n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b) != bench._code_only(c)
    assert bench.kernel_source_digest("bwd_main") != bench.kernel_source_digest("fwd")
    assert bench.kernel_source_digest("no_such_kernel") is None


def test_splitkv_work_counts():
    # decode: 8 x 32 heads, one query row against 32768 keys, d = 128
    flops, nbytes = bench.splitkv_work(8, 32, 1, 32768, 128)
    assert flops == 4 * 256 * 32768 * 128
    kv = 2 * 256 * 32768 * 128 * 2          # K and V in bf16
    assert nbytes == kv + 2 * 256 * 128 * 2 + 256 * 4  # + Q and O rows in bf16, LSE in fp32
    assert abs(kv - 4.295e9) < 1e6           # the 4.30 GB the traffic capture reads


def test_visible_counts_match_the_element_mask():
    from oracle.tiled import visible_mask
    rng = np.random.default_rng(3)
    n, tile = 45, 8
    T = (n + tile - 1) // tile
    bm = (rng.random((T, T)) < 0.5).astype(np.uint8)
    rows = np.arange(n)
    for causal in (False, True):
        for kl in (None, 0, 17, n):
            for mask in (None, bm):
                vis = visible_mask(n, causal, kl, mask, tile)
                got = bench.row_visible_counts(n, rows, causal, kl, mask, tile=tile)
                assert np.array_equal(got, vis.sum(axis=1)), (causal, kl, mask is None)
    # whole workload: lengths per sequence, heads multiply
    kv = np.array([100, 300], np.int32)
    assert bench.useful_score_pairs(300, False, kv, None, 2, 3) == 3 * 300 * (100 + 300)
    assert bench.useful_score_pairs(300, True, None, None, 1, 2) == 2 * 300 * 301 // 2


def test_oracle_extrapolation_doubles_the_row_pass():
    # the column pass is counted at the row pass's cost per visible pair
    assert bench.extrapolated_oracle_seconds(2.0, 1000, 50000) == pytest.approx(200.0)


def test_clock_windows_pick_their_own_samples():
    s = bench.ClockSampler(0)
    line = "0, {}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {}"
    s.samples = [(1.0, line.format(2000, "Not Active")), (2.0, line.format(1900, "Active")),
                 (3.0, line.format(2070, "Not Active")), (4.0, line.format(2070, "Not Active"))]
    a = s.window(0.5, 2.5)
    assert a["samples"] == 2 and a["sm_mhz"] == 1950 and a["reasons"] == ["sw_power_cap"]
    b = s.window(2.5, 5.0)
    assert b["samples"] == 2 and b["sm_mhz"] == 2070 and b["reasons"] == []
    assert s.window(10, 11)["samples"] == 0


def test_standard_attention_is_the_definition_in_fp64():
    # the comparison leg's arithmetic, run on the CPU in float64, is the oracle's definition
    import torch
    import oracle
    from io_aware_exact_attention_gb300 import inputs
    for causal in (False, True):
        inp = inputs.make_inputs(1, 2, 70, 16, seed=5, causal=causal, with_dout=False)
        q, k, v = (torch.from_numpy(np.asarray(getattr(inp, n), np.float64)) for n in ("q", "k", "v"))
        o = bench.standard_attention(torch, q, k, v, inp.scale, causal).numpy()
        ref_o, _ = oracle.attention_forward(inp.q, inp.k, inp.v, inp.scale, causal=causal)
        np.testing.assert_allclose(o, ref_o, rtol=1e-11, atol=1e-12)


def test_block_mask_legs_count_visited_tiles():
    from io_aware_exact_attention_gb300 import inputs
    inp = inputs.make_inputs(1, 2, 512, 64, seed=3, block_mask=dict(band=0, global_cols=0, frac=0.0))
    pairs = bench.visited_tile_pairs(512, False, None, inp.block_mask, 1, 2)
    assert pairs == 2 * 4  # the diagonal tiles only
    ms = {"fwd": 1.0, "bwd_preprocess": 0.1, "bwd_main": 2.0, "bwd_postprocess": 0.1, "stages_sum": 3.2,
          "step": 3.2, "wall_s": 1.0, "launch": "api calls", "steps": 10, "window": (0.0, 1.0)}
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "test"}
    rep = bench.leg_report(inp, ms, pairs, peaks, bench.parse_clock_lines([]))
    alg = bench.algorithmic_flops(pairs, 64)
    assert rep["fwd_tflops"] == round(alg["fwd"] / 1e-3 / 1e12, 2)
    assert rep["dense_equivalent"]["fwd_tflops"] == round(bench.formula_fwd_flops(1, 2, 512, 64, False) / 1e-3 / 1e12, 2)
    assert rep["flops_per_step"]["formula_fwd"] == bench.formula_fwd_flops(1, 2, 512, 64, False)
