"""Shared helpers for the GPU parity tests (torch <-> numpy, error checks)."""
import numpy as np

from oracle import oracle as orc

TOL_F32 = 1e-5   # relative Frobenius per object, fp32-input workloads
TOL_BF16 = 5e-3  # relative Frobenius per object, bf16-input workloads (oracle reads the same bf16 values)


def torch():
    import torch as t
    return t


def dev(x, dtype="f32"):
    """numpy float32 (bf16 values already rounded when dtype='bf16') -> CUDA tensor."""
    t = torch()
    if x is None:
        return None
    a = t.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        a = a.to(t.bfloat16)  # exact: the values are bf16-representable
    return a.cuda()


def host(x):
    return None if x is None else x.detach().float().cpu().numpy().astype(np.float64)


def gdn_T64(T, T_exp):
    """GPU mantissa + exponent -> float64 T_C."""
    return orc.scaled_to_f64(T.detach().cpu().numpy(), T_exp.detach().cpu().numpy())


def assert_rel(x, ref, tol, axes=(-2, -1), what=""):
    r = orc.rel_fro(x, ref, axes)
    worst = float(np.max(r)) if r.size else 0.0
    assert worst <= tol, f"{what}: max relative Frobenius error {worst:.3e} > {tol:.1e}"
    return worst


def seam_inputs_from(inputs, token_index):
    """Gather rows `token_index` (host int array) of the per-token arrays."""
    out = {}
    for key in ("q", "k", "v", "alpha", "beta", "g"):
        if key in inputs and inputs[key] is not None:
            out[key] = np.ascontiguousarray(inputs[key][:, token_index])
    return out
