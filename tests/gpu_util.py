"""Helpers shared by the GPU parity tests: device upload, the tolerance bar, and the
all-rows check of full-size results.

Tolerance (floating point): each element satisfies, before the output cast,
    |D - D_ref| <= 1e-2 * sqrt(K / 256) * (|A||B|)_ij + 1e-6
and the cast adds at most half an ulp of the output type, so the test allows
u_out * |D_ref| on top (u_out = 2^-8 BF16, 2^-11 FP16, 0 FP32).  The relative
Frobenius error of the result before the cast, ||D - D_ref||_F / ||D_ref||_F, is at
most 1e-3 (FP16/BF16 inputs) or 2e-2 (FP8 inputs); a cast to BF16/FP16 moves each
element by at most u_out * |D|, so on a cast output the test allows
(bar + u_out * (1 + bar)) * ||D_ref||_F.  An FP32 output carries no allowance.
The integer path is compared bit for bit.
"""
import numpy as np
import torch

U_OUT = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}
FROB = {"f16": 1e-3, "bf16": 1e-3, "e4m3": 2e-2}


def dev():
    return torch.device("cuda:0")


def up(a):
    """Upload a numpy array to cuda:0 keeping its raw bytes (uint16 -> int16 view)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def out_tensor(M, ldd, out, fill=float("nan")):
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out]
    return torch.full((M, ldd), fill, dtype=dt, device=dev())


def out_code(out):
    import linear_layer_gb300 as ll
    return {"f32": ll.OUT_F32, "bf16": ll.OUT_BF16, "f16": ll.OUT_F16}[out]


def check_close(D, ref, absab, K, out, in_kind, what=""):
    D = np.asarray(D, dtype=np.float64)
    bound = 1e-2 * np.sqrt(max(K, 1) / 256.0) * absab + 1e-6 + U_OUT[out] * np.abs(ref)
    err = np.abs(D - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d elements outside tolerance, e.g. %s: got %s want %s bound %s" % (
            what, int(bad.sum()), idx.tolist(), D[tuple(idx[0])], ref[tuple(idx[0])],
            bound[tuple(idx[0])]))
    nref = np.linalg.norm(ref)
    if nref > 0:
        rel = np.linalg.norm(D - ref) / nref
        bar = FROB[in_kind] + U_OUT[out] * (1.0 + FROB[in_kind])
        assert rel <= bar, "%s: relative Frobenius error %g > %g" % (what, rel, bar)


def check_all_rows(D, oracle_rows, M, N, K, out, in_kind, what="", chunk=512):
    """Compare every element of D[:M, :N] with the oracle, `chunk` rows at a time
    (oracle_rows(rows) -> (ref, absab) for those rows), at the per-element bound of
    check_close; the relative Frobenius bar is applied to the whole matrix."""
    D = np.asarray(D)
    num = 0.0
    den = 0.0
    for r0 in range(0, M, chunk):
        rows = np.arange(r0, min(M, r0 + chunk), dtype=np.int32)
        ref, absab = oracle_rows(rows)
        Dc = D[rows, :N].astype(np.float64)
        bound = 1e-2 * np.sqrt(max(K, 1) / 256.0) * absab + 1e-6 + U_OUT[out] * np.abs(ref)
        err = np.abs(Dc - ref)
        bad = ~(err <= bound)
        if bad.any():
            idx = np.argwhere(bad)[:5]
            i, j = idx[0]
            raise AssertionError("%s: %d elements outside tolerance in rows %d..%d, e.g. (%d, %d): got %s "
                                 "want %s bound %s" % (what, int(bad.sum()), r0, rows[-1], r0 + i, j, Dc[i, j],
                                                       ref[i, j], bound[i, j]))
        num += float(np.sum((Dc - ref) ** 2))
        den += float(np.sum(ref ** 2))
    if den > 0:
        rel = np.sqrt(num / den)
        bar = FROB[in_kind] + U_OUT[out] * (1.0 + FROB[in_kind])
        assert rel <= bar, "%s: relative Frobenius error %g > %g" % (what, rel, bar)


def assert_fully_written(tD, M, N, what=""):
    """D was pre-filled with NaN and the inputs are finite: every element of D[:M, :N] must
    have been written (a skipped tile would leave NaN)."""
    import torch
    nan = torch.isnan(tD[:M, :N].float())
    if bool(nan.any()):
        idx = torch.nonzero(nan)[:5].tolist()
        raise AssertionError("%s: %d elements of D never written, e.g. %s" % (what, int(nan.sum()), idx))
