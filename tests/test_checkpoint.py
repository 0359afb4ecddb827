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
