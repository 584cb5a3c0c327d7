"""Host logic of bench.py that needs no GPU: the replica plumbing over two
gloo ranks (barrier, max over ranks, per-rank seeds), byte counts, the
traffic lookup and the reference arm's JSON line on a tiny workload."""
import json
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from gqa_kv_cache_append_gb300.inputs import layer_bytes, seq_lens_for, workload


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, float(10 + rank * 5))
    q.put((rank, m, bench.replica_seed(3, rank)))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
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
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] != res[1][2]


def test_single_process_needs_no_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 2.5) == 2.5


def test_step_bytes_llama3_shape():
    cfg = workload("llama3_70b_b32_m8192")
    lens = seq_lens_for(cfg)
    sb = bench.step_bytes(cfg, lens)
    # K and V rows of 8 KV heads x 8192 positions x 32 sequences, plus q and out
    assert sb["attn_per_layer"] == 32 * 8 * 8192 * 2 * 128 * 2 + 2 * 32 * 64 * 128 * 2
    assert sb["attn_per_layer"] == layer_bytes(cfg, lens) == 1074790400
    assert sb["step"] == 80 * (sb["attn_per_layer"] + 4 * 32 * 8 * 128 * 2)


def test_ragged_lengths_bytes():
    cfg = workload("qwen25_7b_b64_ragged")
    lens = seq_lens_for(cfg)
    assert int(lens.sum()) == 1203078
    assert layer_bytes(cfg, lens) == 1203078 * 4 * 2 * 128 * 2 + 2 * 64 * 28 * 128 * 2


def test_traffic_lookup_requires_matching_source(tmp_path, monkeypatch):
    src = tmp_path / "decode_tc.cu"
    src.write_text("kernel v1")
    (tmp_path / "gqa_device.cuh").write_text("header v1")
    prof = tmp_path / "profiles"
    prof.mkdir()
    import hashlib
    h = hashlib.sha256(b"kernel v1header v1").hexdigest()
    assert bench.kernel_source_hash(str(src)) == h
    (prof / "decode_tc_w.md").write_text(f"source_sha256: {h}\ntraffic_bytes_per_launch: 1234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic(str(src), "w") == 1234
    (tmp_path / "gqa_device.cuh").write_text("header v2")
    assert bench.profiled_traffic(str(src), "w") is None   # the header changed
    (tmp_path / "gqa_device.cuh").write_text("header v1")
    assert bench.profiled_traffic(str(src), "w") == 1234
    src.write_text("kernel v2")
    assert bench.profiled_traffic(str(src), "w") is None
    # the summary is looked up by the kernel's own name
    other = tmp_path / "decode_simt.cu"
    other.write_text("kernel v1")
    assert bench.profiled_traffic(str(other), "w") is None


def test_reference_arm_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                "--workload", "mqa_f32_b1_h8_d64_m256", "--ref-seconds", "2"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == bench.host_cores()


def test_oracle_sample_uses_every_core():
    cfg = workload("mqa_f32_b1_h8_d64_m256")
    gbs, wall, units, nbytes, cores = bench.oracle_sample(cfg, target_s=0.3)
    assert cores == bench.host_cores() and gbs > 0 and wall > 0
    # every worker ran whole units: bytes are a multiple of one unit's bytes
    one = (256 * cfg.g + cfg.h) * (cfg.d + cfg.dv) * cfg.elt
    assert nbytes % one == 0 and nbytes // one == units // cfg.g


@pytest.mark.parametrize("nl", [1, 2, 3, 4, 5, 8, 9, 28, 80, 81, 4011])
def test_copy_groups_cover_every_layer(nl):
    """The end-to-end copy schedule: both lists tile 0..nl in order; the
    inputs take at most three groups, the first layer's alone; the outputs
    at most about ten plus the last layer alone."""
    ins, outs = bench.copy_groups(nl)
    for groups in (ins, outs):
        assert groups[0][0] == 0 and groups[-1][1] == nl
        assert all(a < z for a, z in groups)
        assert all(groups[i][1] == groups[i + 1][0] for i in range(len(groups) - 1))
    assert ins[0] == (0, 1) and len(ins) <= 3
    assert outs[-1] == (nl - 1, nl) and len(outs) <= 12
    if nl == 80:
        assert ins == [(0, 1), (1, 4), (4, 80)]
        assert len(outs) == 11 and outs[0] == (0, 8) and outs[-2] == (72, 79)
