"""Host logic of bench.py for N > 1 (independent replicas): rendezvous,
barrier, max-over-ranks timing and the whole-job aggregate, run as two `gloo`
processes on the CPU."""

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    dist = bench.dist_init(w, "gloo")
    bench.dist_barrier(dist)
    # each replica times its own steps; the job's time is the slowest rank's
    my_ms = 10.0 + 5.0 * rank
    ms = bench.dist_max(dist, my_ms)
    flops_per_replica = 1e12
    value = w * flops_per_replica / (ms * 1e-3) / 1e12
    rec = bench.make_record(value=value, n_gpus=w, steps=3, warmup=3, ms_per_step=ms,
                            config={"workload": "test"}, extra={"gpu_launches": 12})
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(rec, f)
    dist.destroy_process_group()


def test_two_rank_replicas_take_max_time(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    recs = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for rec in recs:
        assert rec["ms_per_step"] == 15.0                    # max over ranks
        assert rec["value"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)   # whole job
        assert rec["n_gpus"] == 2 and rec["scaling"] == "weak"
        for key in ("metric", "unit", "steps", "warmup", "higher_is_better", "vs_baseline",
                    "dtype", "data", "config"):
            assert key in rec


def test_single_rank_needs_no_process_group():
    assert bench.dist_init(1, "gloo") is None
    assert bench.dist_max(None, 3.5) == 3.5


def test_peaks_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0


def test_quantize_roofline_counts_fp32_in_and_q8_0_out():
    """q8kv_quantize of K and V moves 256 B of fp32 in and 68 B of Q8_0 out per
    64-value head row: 2 * B * M * H * 324 bytes per step."""
    import bench
    rec = bench.quantize_record(1, 65536, 32, 64, 0.2, {"hbm_gbs": 6795.1}, "measured")
    assert rec["algorithmic_bytes"] == 2 * 65536 * 32 * 324
    assert abs(rec["achieved"] - rec["algorithmic_bytes"] / 0.2e-3 / 1e9) < 1e-6
    assert abs(rec["frac"] - rec["achieved"] / 6795.1) < 1e-12
    assert rec["bound"] == "hbm" and rec["unit"] == "GB/s"


def test_step_bytes_of_the_smallest_workload():
    """m512 (1 x 512 tokens, 32 heads, chunks of 128): quantise 2 x 324 B, init
    264 B and finalise 388 B per state row, and per chunk 656 B per state row
    at or after the chunk start plus 136 B per chunk key and head."""
    import bench
    from chunked_prefill_attention_gb300 import workloads as W
    rows = 32 * 512
    chunks = sum(32 * (512 - s0) * 656 + 32 * 128 * 136 for s0 in (0, 128, 256, 384))
    assert bench.step_hbm_bytes(W.WORKLOADS["m512"]) == rows * (2 * 324 + 264 + 388) + chunks


def test_split_keys_for_whole_waves():
    """Range lengths for the split launch: whole waves of one CTA per SM."""
    from chunked_prefill_attention_gb300.q8attn import split_keys_for
    # 32 heads on 152 SMs: four waves = 608 CTAs = 19 ranges
    n = split_keys_for(32, 1048576, 152)
    assert n == 55296 and n % 128 == 0 and -(-1048576 // n) == 19
    # one head on 152 SMs: one wave of 152 ranges
    n = split_keys_for(1, 1048576, 152)
    assert n % 128 == 0 and -(-1048576 // n) == 152
    # 8 heads over 65,536 keys: one wave of 19 ranges of 3,456 keys
    n = split_keys_for(8, 65536, 152)
    assert n == 3456 and -(-65536 // n) * 8 == 152
    # 9 heads: no whole number of waves within eight (152 w is a multiple of 9
    # only from w = 9), and ranges that would be too short: 8,192
    assert split_keys_for(9, 1 << 20, 152) == 8192
    assert split_keys_for(1, 100000, 152) == 8192
    with pytest.raises(ValueError):
        split_keys_for(0, 10, 152)
