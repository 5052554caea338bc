"""Shared helpers of the GPU parity tests: metrics, transfers, oracle runs."""
import numpy as np

REL_TOL = 1e-2          # relative Frobenius error bound on O, O', dQ, dK, dV
COS_TOL = 0.999         # cosine similarity bound
LSE_TOL = 1e-3          # max abs error of the natural-log LSE
TILE_ROWS = 128         # rows per block of the per-tile checks (the kernels' tile)


def rel_cos(got, ref):
    a = np.asarray(got, np.float64).ravel()
    b = np.asarray(ref, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if nb == 0:
        return (0.0 if na == 0 else np.inf), (1.0 if na == 0 else 0.0)
    rel = np.linalg.norm(a - b) / nb
    cos = float(a @ b / (na * nb)) if na > 0 else 0.0
    return rel, cos


def assert_close(name, got, ref, rel_tol=REL_TOL, cos_tol=COS_TOL, tile=TILE_ROWS):
    """The bounds over the whole tensor, then over every `tile`-row block of
    each head (axis -2 holds the rows), the granularity at which the kernels
    own their outputs: one wrong row or tile cannot hide under the norm of
    the rest. A block whose reference is exactly zero must be exactly zero."""
    rel, cos = rel_cos(got, ref)
    assert rel <= rel_tol and cos >= cos_tol, f"{name}: rel={rel:.3e} cos={cos:.6f}"
    assert_tiles(name, got, ref, rel_tol, cos_tol, tile)
    return rel, cos


def assert_tiles(name, got, ref, rel_tol=REL_TOL, cos_tol=COS_TOL, tile=TILE_ROWS):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} != {r.shape}"
    if g.ndim < 2:
        return
    n = g.shape[-2]
    g = g.reshape(-1, n, g.shape[-1])
    r = r.reshape(-1, n, r.shape[-1])
    for h in range(g.shape[0]):
        for t0 in range(0, n, tile):
            rel, cos = rel_cos(g[h, t0:t0 + tile], r[h, t0:t0 + tile])
            assert rel <= rel_tol and cos >= cos_tol, \
                f"{name}: head {h} rows [{t0}, {min(n, t0 + tile)}): rel={rel:.3e} cos={cos:.6f}"


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
