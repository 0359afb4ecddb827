"""The benchmark's algorithmic byte counts for the Llama-3-8B layer, against
sums worked out by hand from the layer shapes (q, o 4096 x 4096; k, v
1024 x 4096; gate, up 14336 x 4096; down 4096 x 14336), E8 codes with tile 256:
quantize reads 2 B of bf16 and writes a 1 B code per weight plus a 4 B scale
per 256 weights and reads each matrix's signs (one byte per column); a GEMV
call reads codes, scales and signs, its activation once per group (bf16) and
writes fp32 y."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

WEIGHTS = 2 * 4096 * 4096 + 2 * 1024 * 4096 + 2 * 14336 * 4096 + 4096 * 14336   # 218 103 808
SIGN_BYTES = 6 * 4096 + 14336                                                     # per-matrix columns
OUT_ROWS = 4096 + 1024 + 1024 + 4096 + 14336 + 14336 + 4096                      # 43 008
# one activation row per group: q/k/v and o and gate/up read 4096 columns, down 14336
X_COLS = 4096 + 4096 + 4096 + 14336


def test_layer_weight_count():
    assert WEIGHTS == 218_103_808
    assert sum(r * c for _, r, c, _ in bench.layer_shapes()) == WEIGHTS


def test_quantize_bytes_of_the_layer():
    q, _, _ = bench.step_bytes(bench.layer_shapes())
    # 3 B per weight + 4 B per 256 weights = 3 + 1/64 B per weight
    expect = WEIGHTS * 3 + WEIGHTS // 64 + SIGN_BYTES
    assert expect == 657_758_208
    assert q == expect


def test_gemv_bytes_of_the_layer_per_batch():
    _, per_b, total = bench.step_bytes(bench.layer_shapes())
    codes_scales = WEIGHTS + WEIGHTS // 64
    for b in (1, 4, 16):
        expect = codes_scales + SIGN_BYTES + b * X_COLS * 2 + b * OUT_ROWS * 4
        assert per_b[b] == expect, (b, per_b[b], expect)
    assert per_b[1] == 221_775_872
    assert total == 657_758_208 + sum(per_b.values())


def test_groups_share_one_activation():
    shapes = bench.layer_shapes()
    groups = bench.layer_groups(shapes)
    names = [[shapes[i][0] for i in g] for g in groups]
    assert names == [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    for g in groups:
        assert len({shapes[i][2] for i in g}) == 1   # one column count (the shared x) per group
