"""CPU checks of bench.py's measurement arithmetic: the algorithmic bytes per expert that the
HBM roofline divides by, and the source fingerprint that keys recorded DRAM traffic."""

from dataclasses import replace

import bench
from synth import LAYERS


def test_expert_bytes_per_format():
    glm = LAYERS["glm52"]
    gu, d = bench.expert_bytes(glm)
    # one GLM-shaped int4-g32 expert: 18,874,368 B of codes + 2,359,296 B of fp16 scales
    assert gu + d == 21_233_664
    assert gu == 2 * d
    n_gu, n_d = bench.expert_bytes(LAYERS["glm52_nvfp4"])
    assert (n_gu, n_d) == (gu + 4, d + 4)          # same code and scale bytes + fp32 tensor scale
    H, I = glm.hidden, glm.inter
    for fmt, bits in (("int8_row", 8), ("int4_row", 4), ("int2_row", 2)):
        r_gu, r_d = bench.expert_bytes(replace(glm, weight_format=fmt, shared_format=fmt))
        assert r_gu == 2 * I * (H * bits // 8 + 4) and r_d == H * (I * bits // 8 + 4)


def test_fingerprint_ignores_comments_only():
    code = "int f(int x) {\n  return x + 1;  // add one\n}\n/* block\n comment */\n"
    same = "int f(int x) {\n  return x + 1;\n}\n\n// another comment\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.source_fingerprint(code) == bench.source_fingerprint(same)
    assert bench.source_fingerprint(code) != bench.source_fingerprint(other)
