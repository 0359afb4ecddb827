"""Save / load of quantized tensors (host only)."""
import numpy as np
import pytest

import oracle as O
from synthetic import gaussian_matrix


def test_round_trip(tmp_path):
    torch = pytest.importorskip("torch")
    import lattice_vq_weight_gb300 as L
    W = gaussian_matrix(8, 512, 0.02, 3)
    d = O.splitmix64_signs(4, 512)
    q = O.quantize(W, "e8", 256, d, 0.25)
    codes = torch.from_numpy(q.codes.astype(np.int8))
    scales = torch.from_numpy(q.scales)
    signs = torch.from_numpy(d.astype(np.int8))
    path = tmp_path / "w.lq"
    L.save_quantized(path, codes, scales, signs, "e8", 256, 4, 0.25)
    back = L.load_quantized(path)
    assert back["lattice"] == "e8" and back["tile"] == 256 and back["seed"] == 4 and back["beta"] == 0.25
    assert torch.equal(back["codes"], codes) and torch.equal(back["scales"], scales)
    assert torch.equal(back["signs"], signs)
    torch.save({"format": "other"}, tmp_path / "x.lq")
    with pytest.raises(ValueError):
        L.load_quantized(tmp_path / "x.lq")


def test_round_trip_with_row_scales_and_dither_seed(tmp_path):
    """Per-row bf16 scales and a dither seed travel with the codes; an older file
    without those fields reads as float32 tile scales and no dither."""
    torch = pytest.importorskip("torch")
    import lattice_vq_weight_gb300 as L
    from oracle import scale_formats as F
    W = gaussian_matrix(6, 512, 0.02, 5)
    d = O.splitmix64_signs(6, 512)
    q = F.quantize_formatted(W, "d4", 128, d, 0.25, "row_bf16")
    codes = torch.from_numpy(q.codes.astype(np.int8))
    scales = torch.from_numpy(q.scales.astype(np.float32)).to(torch.bfloat16)
    signs = torch.from_numpy(d.astype(np.int8))
    L.save_quantized(tmp_path / "r.lq", codes, scales, signs, "d4", 128, 6, 0.25, scale_format="row_bf16",
                     dither_seed=2 ** 63 + 1)
    back = L.load_quantized(tmp_path / "r.lq")
    assert back["scale_format"] == "row_bf16" and back["dither_seed"] == 2 ** 63 + 1
    assert back["scales"].dtype == torch.bfloat16 and torch.equal(back["scales"], scales)
    assert torch.equal(back["codes"], codes)
    old = {k: v for k, v in back.items() if k not in ("scale_format", "dither_seed")}
    old["scales"] = torch.zeros((6, 4), dtype=torch.float32)
    torch.save(old, tmp_path / "old.lq")
    again = L.load_quantized(tmp_path / "old.lq")
    assert again["scale_format"] == "tile_f32" and again["dither_seed"] is None
    with pytest.raises(ValueError):
        L.save_quantized(tmp_path / "z.lq", codes, scales, signs, "d4", 128, 6, 0.25, scale_format="nope")
