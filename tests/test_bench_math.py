"""The bench's algorithmic work (the numerators of every roofline fraction)
against the closed forms: per token 6·K·d·f + 2·d·E FLOPs for the layer and
4·K·d·f for the gate/up GEMM; per touched expert 3·d·f weights streamed
(2 bytes each in bf16, 1 in e4m3 plus fp32 column scales).  And the hash that
keys the recorded DRAM traffic to a kernel's code ignores comments only."""
from __future__ import annotations

import pathlib

import pytest

import bench

MIX = dict(d=4096, f=14336, E=8, K=2)


def test_prefill_flops_and_bytes():
    c = dict(T=4096, **MIX)
    flops, gu_flops, bytes_step, gu_bytes = bench.algorithmic(c, n_touched=8)
    assert flops == 4096 * (2 * 6 * 4096 * 14336 + 2 * 4096 * 8)
    assert flops / 4096 == pytest.approx(704.7e6, rel=1e-4)          # 704.7 MFLOP per token
    assert gu_flops == 4096 * 2 * 4 * 4096 * 14336                   # 469.8 MFLOP per token
    assert gu_flops / 4096 == pytest.approx(469.8e6, rel=1e-4)
    per_expert = 3 * 4096 * 14336 * 2
    assert per_expert == pytest.approx(352.3e6, rel=1e-4)             # 352.3 MB per touched expert
    assert bytes_step == 8 * per_expert + 2 * 4096 * 8 + 2 * 4096 * 4096 * 2
    assert gu_bytes == 8 * (2 * 4096 * 14336 * 2 + 2 * 14336 * 4)


def test_decode_and_fp8_bytes():
    _, _, b1, gu1 = bench.algorithmic(dict(T=1, **MIX), n_touched=2)
    assert gu1 == 2 * (2 * 4096 * 14336 * 2 + 2 * 14336 * 4)         # 469.8 MB + column scales
    _, _, b8, gu8 = bench.algorithmic(dict(T=1, fp8=True, **MIX), n_touched=2)
    assert gu8 == 2 * (2 * 4096 * 14336 * 1 + 2 * 14336 * 4)
    assert b8 == 2 * (3 * 4096 * 14336 + 3 * 14336 * 4 + 4096 * 4) + 2 * 4096 * 8 + 2 * 1 * 4096 * 2


def test_code_hash_ignores_comments_only(tmp_path: pathlib.Path):
    a = tmp_path / "a.cu"
    a.write_text("int f() {  // one\n  return 1;\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("// header\nint f() {\n\n  return 1;  // other words\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f() {\n  return 2;\n}\n")
    assert bench.code_sha256(a) == bench.code_sha256(b)
    assert bench.code_sha256(a) != bench.code_sha256(c)


def test_recorded_traffic_follows_the_kernel_hash():
    """The DRAM bytes recorded by an ncu capture are reported only while the
    kernel's code still hashes to the recorded value; otherwise null."""
    import re
    root = bench.ROOT / "sparse_mixture_experts_55_b300" / "csrc"
    for src, summary, key in ((root / "gemm_tc.cu", "gate_up_gemm_traffic.md", "prefill_traffic_bytes_per_launch"),
                              (root / "gemm_bwd.cu", "bwd_gemm_traffic.md", "train_wgrad_w13_traffic_bytes_per_launch")):
        text = (bench.ROOT / "profiles" / summary).read_text()
        recorded = re.search(r"code_sha256:\s*([0-9a-f]{64})", text).group(1)
        value = float(re.search(rf"{key}:\s*([0-9.eE+]+)", text).group(1))
        got = bench.traffic_from_profiles(src, key, summary)
        assert got == (value if bench.code_sha256(src) == recorded else None)
