"""bench.py's workload arithmetic (no GPU): algorithmic bytes and FLOPs
against brute-force counts, and the extend split chooser's rules."""
import types

import bench


def _p(batch, Hq, Hkv, D, lens):
    return types.SimpleNamespace(batch=batch, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D,
                                 group=Hq // Hkv,
                                 seq_lens=types.SimpleNamespace(tolist=lambda: list(lens)))


def test_extend_flops_brute_force():
    lens, qo = [10, 7, 33], [3, 7, 1]
    p = _p(3, 8, 2, 64, lens)
    pairs = 0
    for L, n in zip(lens, qo):
        for i in range(n):
            for t in range(L):
                pairs += t <= L - n + i  # keys each new token attends
    assert bench.extend_flops(lens, qo, p) == 4 * 64 * 8 * pairs


def test_extend_bytes():
    lens, qo = [10, 7], [3, 7]
    p = _p(2, 8, 2, 64, lens)
    kv = sum(lens) * 2 * 64 * 2 * 2  # K and V of every context token, bf16
    qout = sum(qo) * 8 * 64 * 2 * 2  # q and out, bf16
    assert bench.extend_bytes(lens, qo, p) == kv + qout


def test_decode_algorithmic_bytes():
    lens = [100, 7]
    p = _p(2, 32, 8, 128, lens)
    want = sum(lens) * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 * 2
    assert bench.algorithmic_bytes(lens, p) == want


def test_traffic_record_applies_only_to_its_kernel_source(tmp_path, monkeypatch):
    # The committed DRAM traffic per launch is reported only while the decode
    # kernel's sources hash to the recorded value, scaled by the algorithmic
    # bytes of the two launches; another source, another workload or a
    # missing record gives None.
    import json
    import os
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"w": {"kernel_src_sha1": "abc", "dram_bytes_per_launch": 1100.0,
                 "algorithmic_bytes_per_launch": 1000.0}}
    (prof / "decode_attn_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("abc", "w", 2000.0) == 2200.0
    assert bench.traffic_for("abd", "w", 2000.0) is None
    assert bench.traffic_for("abc", "other", 2000.0) is None
    os.remove(prof / "decode_attn_traffic.json")
    assert bench.traffic_for("abc", "w", 2000.0) is None


def test_kernel_source_hash_covers_the_decode_sources(tmp_path, monkeypatch):
    # The hash changes with decode*.cu and the shared headers, not with the
    # extend kernel or the host entry points.
    csrc = tmp_path / "paged_kv_decode_bind_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("decode_mma.cu", "merge.cuh", "extend_mma.cu", "pkv_api.cu"):
        (csrc / name).write_text(name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_src_hash()
    for name, moves in (("extend_mma.cu", False), ("pkv_api.cu", False),
                        ("decode_mma.cu", True), ("merge.cuh", True)):
        (csrc / name).write_text(name + " changed")
        assert (bench.kernel_src_hash() != h0) == moves, name
        (csrc / name).write_text(name)
