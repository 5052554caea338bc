"""Shared helpers of the GPU parity tests: metrics, transfers, oracle runs."""
import numpy as np

REL_TOL = 1e-2          # relative Frobenius error bound on O, O', dQ, dK, dV
COS_TOL = 0.999         # cosine similarity bound
LSE_TOL = 1e-3          # max abs error of the natural-log LSE


def rel_cos(got, ref):
    a = np.asarray(got, np.float64).ravel()
    b = np.asarray(ref, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if nb == 0:
        return (0.0 if na == 0 else np.inf), (1.0 if na == 0 else 0.0)
    rel = np.linalg.norm(a - b) / nb
    cos = float(a @ b / (na * nb)) if na > 0 else 0.0
    return rel, cos


def assert_close(name, got, ref, rel_tol=REL_TOL, cos_tol=COS_TOL):
    rel, cos = rel_cos(got, ref)
    assert rel <= rel_tol and cos >= cos_tol, f"{name}: rel={rel:.3e} cos={cos:.6f}"
    return rel, cos


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev(a):
    import torch
    return to_dev(np.asarray(a, np.float32), torch.bfloat16)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def round_bf16(a):
    """Round float64 values to BF16 (ties to even) as float64."""
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
