"""The .fp8w file: a quantised weight (e4m3 codes and their scales) with a
format tag, so that quantisation runs once and serving loads its result.

The pages quantise at load time from a bf16/fp32 checkpoint and tag fp8
data by its format (e4m3fn, e8m0fnu); they define no file.  This one is
plain and little-endian:

    offset  size  field
    0       4     magic b"FP8W"
    4       4     version (1)
    8       4     scale kind: 0 one fp32 per row [n]; 1 fp32 per group
                  [n, k / group]; 2 E8M0 bytes per 32 codes [n, k / 32]
    12      4     code format: 0 OCP e4m3fn
    16      8     n (rows, output channels)
    24      8     k (codes a row)
    32      8     group (0 for kind 0, 32 for kind 2)
    40      4     CRC-32 of the codes
    44      4     CRC-32 of the scales
    48      16    zero
    64      n*k   codes, row-major
    ...           scales, row-major, from the next multiple of 64

Writing and reading use host memory only; load() copies to the device
asked for.  Every field, both sizes and both checksums are checked on
load, and any mismatch raises.
"""
import os
import struct
import zlib

MAGIC = b"FP8W"
VERSION = 1
KIND_ROW, KIND_GROUP, KIND_E8M0 = 0, 1, 2
CODE_E4M3FN = 0
_HDR = struct.Struct("<4sIIIQQQII16x")
assert _HDR.size == 64


class Fp8wFileError(ValueError):
    pass


def _kind_of(codes, scales):
    import torch
    n, k = codes.shape
    if scales.dtype == torch.uint8:
        if scales.dim() != 2 or scales.shape != (n, k // 32) or k % 32:
            raise Fp8wFileError("E8M0 scales must be [n, k / 32]")
        return KIND_E8M0, 32
    if scales.dtype != torch.float32:
        raise Fp8wFileError("scales must be float32 or uint8 (E8M0)")
    if scales.dim() == 1:
        if scales.shape[0] != n:
            raise Fp8wFileError("per-row scales must be [n]")
        return KIND_ROW, 0
    if scales.dim() != 2 or scales.shape[0] != n or scales.shape[1] == 0 or k % scales.shape[1]:
        raise Fp8wFileError("per-group scales must be [n, k / group]")
    return KIND_GROUP, k // scales.shape[1]


def _pad64(x):
    return (x + 63) // 64 * 64


def save(path, codes, scales):
    """Write codes (uint8 [n, k]) and scales (fp32 [n], fp32 [n, k / group]
    or E8M0 uint8 [n, k / 32]), on any device, to path."""
    import torch
    if codes.dtype != torch.uint8 or codes.dim() != 2:
        raise Fp8wFileError("codes must be a 2-D uint8 tensor")
    n, k = codes.shape
    kind, group = _kind_of(codes, scales)
    cb = codes.detach().contiguous().cpu().numpy().tobytes()
    sb = scales.detach().contiguous().cpu().numpy().tobytes()
    hdr = _HDR.pack(MAGIC, VERSION, kind, CODE_E4M3FN, n, k, group, zlib.crc32(cb), zlib.crc32(sb))
    tmp = "%s.tmp%d" % (path, os.getpid())
    with open(tmp, "wb") as f:
        f.write(hdr)
        f.write(cb)
        f.write(b"\0" * (_pad64(64 + len(cb)) - 64 - len(cb)))
        f.write(sb)
    os.replace(tmp, path)


def load(path, device="cuda"):
    """Read a .fp8w file: (codes, scales) on `device`, scales in the dtype and
    shape of their kind."""
    import numpy as np
    import torch
    with open(path, "rb") as f:
        data = f.read()
    if len(data) < 64:
        raise Fp8wFileError("%s: shorter than the header" % path)
    magic, version, kind, code_fmt, n, k, group, ccrc, scrc = _HDR.unpack_from(data, 0)
    if magic != MAGIC:
        raise Fp8wFileError("%s: not an .fp8w file" % path)
    if version != VERSION:
        raise Fp8wFileError("%s: version %d, this reader knows %d" % (path, version, VERSION))
    if code_fmt != CODE_E4M3FN:
        raise Fp8wFileError("%s: unknown code format %d" % (path, code_fmt))
    if n < 1 or k < 1:
        raise Fp8wFileError("%s: empty matrix" % path)
    if kind == KIND_ROW and group == 0:
        sshape, sdt, ssize = (n,), np.float32, 4 * n
    elif kind == KIND_GROUP and group > 0 and k % group == 0:
        sshape, sdt, ssize = (n, k // group), np.float32, 4 * n * (k // group)
    elif kind == KIND_E8M0 and group == 32 and k % 32 == 0:
        sshape, sdt, ssize = (n, k // 32), np.uint8, n * (k // 32)
    else:
        raise Fp8wFileError("%s: bad scale kind %d with group %d" % (path, kind, group))
    s0 = _pad64(64 + n * k)
    if len(data) != s0 + ssize:
        raise Fp8wFileError("%s: %d bytes, the header implies %d" % (path, len(data), s0 + ssize))
    cb = data[64:64 + n * k]
    sb = data[s0:s0 + ssize]
    if zlib.crc32(cb) != ccrc or zlib.crc32(sb) != scrc:
        raise Fp8wFileError("%s: checksum mismatch" % path)
    codes = torch.from_numpy(np.frombuffer(cb, dtype=np.uint8).reshape(n, k).copy())
    scales = torch.from_numpy(np.frombuffer(sb, dtype=sdt).reshape(sshape).copy())
    return codes.to(device), scales.to(device)
