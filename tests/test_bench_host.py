"""Host logic of bench.py: FLOP accounting, the multi-rank control plane (two gloo
ranks on the CPU), the committed-profile parser and the reference arm's JSON."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_37_gb300 import synth  # noqa: E402


def test_flop_accounting():
    w = synth.LONG
    fwd = 4 * 2 * 16 * 8192 * 8192 * 128 / 2
    assert bench.attention_flops(w, backward=False) == fwd
    assert bench.attention_flops(w) == fwd * 3.5
    assert bench.attention_flops(synth.TRAIN) == 4 * 4 * 16 * 2048 * 2048 * 64 * 3.5


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.reduce_max(10.0 + rank, w, torch.device("cpu"))
    out[rank] = m
    dist.destroy_process_group()


def test_two_rank_max_reduce_over_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_profile_traffic_requires_matching_source(tmp_path, monkeypatch):
    import hashlib

    src = tmp_path / "k.cu"
    src.write_text("kernel")
    hdr = tmp_path / "k.cuh"
    hdr.write_text("header")
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = hashlib.sha256(b"kernelheader").hexdigest()
    (prof / "tag.md").write_text(f"- source: `k.cu`, `k.cuh`\n- source_sha256: `{h}`\n- traffic_bytes_per_launch: `1234`\n")
    monkeypatch.setattr(bench, "HERE", str(tmp_path))
    assert bench.profile_traffic("tag") == 1234.0
    hdr.write_text("changed header")
    assert bench.profile_traffic("tag") is None
    hdr.write_text("header")
    src.write_text("changed kernel")
    assert bench.profile_traffic("tag") is None


def test_reference_arm_json_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--workload", "tiny_B1_H1_N256_d64_fp16"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["value"] > 0
