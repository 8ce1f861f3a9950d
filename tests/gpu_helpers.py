"""Shared helpers of the GPU tests: device upload of seeded inputs, calls
through the C ABI binding, and the parity metrics of the tolerance bar."""
from __future__ import annotations

import numpy as np
import torch

from paged_mla_decode_02_gb300 import mla

# Bars for floating-point parity against the float64 oracle.
MAX_ABS = 1e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3


def to_device(x):
    """MLAInputs -> dict of CUDA tensors (bf16 / fp8 bit patterns reinterpreted)."""
    dev = torch.device("cuda")

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def cache(a):
        if x.kv_dtype == "bf16":
            return bf16(a)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(torch.float8_e4m3fn)

    return dict(q_nope=bf16(x.q_nope), q_pe=bf16(x.q_pe), ckv=cache(x.ckv), kpe=cache(x.kpe),
                kv_indices=torch.from_numpy(x.kv_indices.astype(np.int32)).to(dev))


def run_decode(x, d, kernel="default", out_dtype=torch.float32, decoder=None, stream=None):
    """Plan + run one batch through the C ABI; returns (out, lse) as float64 numpy."""
    dec = decoder or mla.MLADecoder(x.batch, x.num_heads, kernel)
    dec.plan(x.kv_indptr, d["kv_indices"], x.kv_len, x.page_size, x.sm_scale, stream=stream)
    out, lse = dec.run(d["q_nope"], d["q_pe"], d["ckv"], d["kpe"], kv_scale=x.kv_scale,
                       out_dtype=out_dtype, stream=stream)
    dec.check_status()
    res = out.double().cpu().numpy(), lse.double().cpu().numpy()
    if decoder is None:
        dec.close()
    return res


def parity(out, lse, ref_out, ref_lse):
    """(max-abs, rel-L2, max |dlse|) over the compared entries."""
    err = out - ref_out
    max_abs = float(np.abs(err).max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref_out))
    rel = float(np.linalg.norm(err) / denom) if denom > 0 else float(np.linalg.norm(err))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(lse)), "lse finiteness differs"
    dl = float(np.abs(lse[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    return max_abs, rel, dl


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    max_abs, rel, dl = parity(out, lse, ref_out, ref_lse)
    assert max_abs <= MAX_ABS and rel <= REL_L2 and dl <= LSE_ABS, (
        f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e} lse={dl:.3e}")
    return max_abs, rel, dl


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float64 -> bf16 -> float64 (torch's CPU cast)."""
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).double().numpy()
