"""The .fp8w file: round trips of every scale kind, and every corruption
refused on load (host only, no GPU)."""
import os

import numpy as np
import pytest
import torch

import fp8_weight_only_gb300 as fw
import oracle
import synthetic


def _kinds():
    w = synthetic.weight_outlier(3, 37, 256)
    c, s = oracle.quantize(w)
    cg, sg = oracle.quantize_grouped(w, 64)
    cm, sm = oracle.quantize_mx(w)
    return {"row": (c, s), "group": (cg, sg), "mx": (cm, sm)}


@pytest.mark.parametrize("kind", ["row", "group", "mx"])
def test_round_trip(tmp_path, kind):
    c, s = _kinds()[kind]
    p = str(tmp_path / "w.fp8w")
    fw.save_fp8w(p, torch.from_numpy(c), torch.from_numpy(s))
    c2, s2 = fw.load_fp8w(p, device="cpu")
    assert c2.dtype == torch.uint8 and np.array_equal(c2.numpy(), c)
    assert s2.dtype == torch.from_numpy(s).dtype and s2.shape == torch.from_numpy(s).shape
    assert np.array_equal(s2.numpy().view(np.uint8), s.view(np.uint8))
    # 64-byte header, codes, padding to a multiple of 64, scales; no temporary left
    assert os.path.getsize(p) == (64 + c.size + 63) // 64 * 64 + s.nbytes
    assert os.listdir(tmp_path) == ["w.fp8w"]


def _saved(tmp_path):
    c, s = _kinds()["group"]
    p = str(tmp_path / "w.fp8w")
    fw.save_fp8w(p, torch.from_numpy(c), torch.from_numpy(s))
    return p, bytearray(open(p, "rb").read())


@pytest.mark.parametrize("offset,what", [(0, "magic"), (4, "version"), (8, "kind"), (12, "code format"),
                                         (100, "a code byte"), (-3, "a scale byte"), (32, "group")])
def test_corruption_is_refused(tmp_path, offset, what):
    p, b = _saved(tmp_path)
    b[offset] ^= 0x5A
    open(p, "wb").write(bytes(b))
    with pytest.raises(fw.Fp8wFileError):
        fw.load_fp8w(p, device="cpu")


def test_truncated_and_extended_files_are_refused(tmp_path):
    p, b = _saved(tmp_path)
    for bad in (bytes(b[:-1]), bytes(b) + b"\0", bytes(b[:40])):
        open(p, "wb").write(bad)
        with pytest.raises(fw.Fp8wFileError):
            fw.load_fp8w(p, device="cpu")


def test_bad_inputs_are_refused_on_save(tmp_path):
    c, s = _kinds()["row"]
    p = str(tmp_path / "w.fp8w")
    with pytest.raises(fw.Fp8wFileError):
        fw.save_fp8w(p, torch.from_numpy(c), torch.from_numpy(s[:-1]))              # wrong row count
    with pytest.raises(fw.Fp8wFileError):
        fw.save_fp8w(p, torch.from_numpy(c), torch.from_numpy(s).double())         # wrong dtype
    with pytest.raises(fw.Fp8wFileError):
        fw.save_fp8w(p, torch.from_numpy(c).float(), torch.from_numpy(s))           # codes not uint8
    with pytest.raises(fw.Fp8wFileError):
        fw.save_fp8w(p, torch.from_numpy(c), torch.zeros((37, 7), dtype=torch.uint8))  # E8M0 not k / 32
    assert not os.path.exists(p)
