"""The NVFP4 inference forward and the NVFP4 packer against the oracle.

Packing is compared bit for bit with oracle.nvfp4_codes (E2M1 codes paired
two per byte, even element in the low nibble, and E4M3 scale bytes). The
attention output O = softmax(scale * Q^ K^T) V (Q^, K^ = the NVFP4 values of
Q and K, V in BF16) is compared with oracle.infer_fwd: relative Frobenius
error <= 1e-2 and cosine >= 0.999 on O, max abs error <= 1e-3 on the LSE.
The long-context shape (B=1 H=16 S=32768 D=128) is checked on sampled query
blocks of the first and last head, in the launch configuration bench.py
times."""
import numpy as np
import pytest

import oracle
from fp4_quantization_aware_gb300 import attnqat, synth
from parity import LSE_TOL, REL_TOL, COS_TOL, bf16_dev, rel_cos

pytestmark = pytest.mark.gpu


def _pack_bytes(codes):
    c = codes.astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def _special_rows(cols):
    """Rows that hit the encoder's edge cases (all BF16-exact)."""
    rows = []
    g = cols // 16
    rows.append(np.zeros(cols, np.float32))                                    # all zero
    rows.append(-np.zeros(cols, np.float32))                                   # all -0
    rows.append(np.full(cols, -1e-3, np.float32))                              # scale rounds to 0, signs kept
    rows.append(np.tile(np.array([6 * 2.0 ** -10] + [0.0] * 15, np.float32), g))  # exactly the zero-scale bound
    rows.append(np.tile(np.array([6 * 2.0 ** -10 * 1.0078125] + [-1e-5] * 15, np.float32), g))  # just above it
    rows.append(np.tile(np.array([3.0e5, -2.5e5] + [1.0] * 14, np.float32), g))  # scale saturates at 448
    rows.append(np.tile(np.linspace(-6, 6, 16, dtype=np.float32), g))          # code midpoints and ties
    rows.append(np.tile(np.array([1e-38, -1e-38] + [2.0 ** -133] * 14, np.float32), g))  # subnormals
    return synth.bf16_round(np.stack(rows))


@pytest.mark.parametrize("cols", [16, 48, 128])
def test_pack_bit_exact(lib, cols):
    import torch
    x = np.concatenate([synth.random_bf16((1000, cols), seed=7 + cols), synth.random_bf16((37, cols), 8, 1e-3),
                        synth.random_bf16((21, cols), 9, 300.0), _special_rows(cols)])
    packed, scales = attnqat.nvfp4_pack(bf16_dev(x))
    torch.cuda.synchronize()
    codes, sc = oracle.nvfp4_codes(x.astype(np.float64), axis=-1)
    np.testing.assert_array_equal(scales.cpu().numpy(), sc)
    np.testing.assert_array_equal(packed.cpu().numpy(), _pack_bytes(codes))


def test_pack_of_attention_shapes(lib):
    """Q of a BHSD tensor packs per row of D = 128 (the layout the kernel reads)."""
    import torch
    w = synth.workload("c2", H=2, Sq=300, Sk=300)
    x = synth.inputs(w)["q"]
    packed, scales = attnqat.nvfp4_pack(bf16_dev(x))
    torch.cuda.synchronize()
    assert tuple(packed.shape) == (1, 2, 300, 64) and tuple(scales.shape) == (1, 2, 300, 8)
    codes, sc = oracle.nvfp4_codes(x.astype(np.float64), axis=-1)
    np.testing.assert_array_equal(scales.cpu().numpy(), sc)
    np.testing.assert_array_equal(packed.cpu().numpy(), _pack_bytes(codes))


CASES = [
    # (B, H, Sq, Sk, causal, structure)
    (1, 2, 256, 256, False, "iid"),
    (1, 2, 384, 384, True, "iid"),
    (2, 1, 300, 300, True, "outlier"),        # ragged tail, causal
    (1, 2, 200, 520, False, "iid"),           # cross-attention, Sq != Sk, ragged
    (1, 1, 1, 1, False, "iid"),               # one query, one key
    (1, 1, 129, 1000, False, "heavy"),
    (1, 3, 640, 640, False, "peaked"),
]


def _case(B, H, Sq, Sk, causal, structure):
    gain = 4.0 if structure == "peaked" else 1.0
    w = synth.Workload("t", B, H, Sq, Sk, 128, causal, 1 / np.sqrt(128),
                       "iid" if structure == "peaked" else structure, gain)
    return w, synth.inputs(w)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_infer_matches_oracle(lib, case):
    import torch
    w, x = _case(*case)
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o, lse = attnqat.infer_fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attnqat.device_status() == 0
    ro, rlse = oracle.infer_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
    rel, cos = rel_cos(o.float().cpu().numpy(), ro)
    assert rel <= REL_TOL and cos >= COS_TOL, f"O rel={rel:.3e} cos={cos:.6f}"
    err = float(np.max(np.abs(lse.cpu().numpy() - rlse)))
    assert err <= LSE_TOL, f"LSE max abs err {err:.3e}"


def test_infer_quantizes_q_and_k(lib):
    """The output follows Q^ K^T, not Q K^T: on outlier channels the two
    oracles differ by far more than the tolerance, and the kernel sits on the
    quantized one."""
    import torch
    w, x = _case(1, 2, 256, 256, False, "outlier")
    o, _ = attnqat.infer_fwd(*(bf16_dev(x[n]) for n in ("q", "k", "v")), causal=False, scale=w.scale)
    torch.cuda.synchronize()
    got = o.float().cpu().numpy()
    rq, _ = oracle.infer_fwd(x["q"], x["k"], x["v"], w.scale, False, quantize=True)
    ru, _ = oracle.infer_fwd(x["q"], x["k"], x["v"], w.scale, False, quantize=False)
    assert rel_cos(rq, ru)[0] > 5 * rel_cos(got, rq)[0]


def test_packed_entry_matches(lib):
    """attnqat_infer_fwd == nvfp4_pack + attnqat_infer_fwd_packed, bit for bit;
    LSE may be omitted."""
    import torch
    w, x = _case(1, 2, 333, 333, True, "iid")
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o1, l1 = attnqat.infer_fwd(q, k, v, causal=True, scale=w.scale)
    qp, qs = attnqat.nvfp4_pack(q)
    kp, ks = attnqat.nvfp4_pack(k)
    o2, l2 = attnqat.infer_fwd_packed(qp, qs, kp, ks, v, causal=True, scale=w.scale)
    o3, l3 = attnqat.infer_fwd_packed(qp, qs, kp, ks, v, causal=True, scale=w.scale, with_lse=False)
    torch.cuda.synchronize()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_infer_repeatable(lib):
    import torch
    w, x = _case(1, 4, 1024, 1024, True, "iid")
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    a = attnqat.infer_fwd(q, k, v, causal=True, scale=w.scale)
    b = attnqat.infer_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_infer_rejects_d64(lib):
    q = bf16_dev(np.zeros((1, 1, 128, 64), np.float32))
    with pytest.raises(attnqat.AttnQatError) as e:
        attnqat.infer_fwd(q, q, q)
    assert e.value.status == 2


def _blocks(n, size=64):
    return [(0, size), ((n // 2) // 16 * 16, (n // 2) // 16 * 16 + size), (n - size, n)]


@pytest.mark.parametrize("causal", [False, True])
def test_ctx32k_sampled(lib, causal):
    import torch
    w = synth.workload("ctx32k", causal=causal)
    x = synth.inputs(w)
    q, k, v = (bf16_dev(x[n]) for n in ("q", "k", "v"))
    o, lse = attnqat.infer_fwd(q, k, v, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attnqat.device_status() == 0
    go, glse = o.float().cpu().numpy(), lse.cpu().numpy()
    report = []
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        qh = oracle.fake_nvfp4(x["q"][b, h].astype(np.float64))
        kh = oracle.fake_nvfp4(x["k"][b, h].astype(np.float64))
        vv = x["v"][b, h].astype(np.float64)
        for r0, r1 in _blocks(w.Sq):
            _, ro, rl = oracle.fwd_rows(qh, kh, vv, w.scale, causal, r0, r1, quantize=False)
            rel, cos = rel_cos(go[b, h, r0:r1], ro)
            err = float(np.max(np.abs(glse[b, h, r0:r1] - rl)))
            report.append(f"({b},{h}) rows [{r0},{r1}): rel={rel:.2e} cos={cos:.6f} lse={err:.2e}")
            assert rel <= REL_TOL and cos >= COS_TOL and err <= LSE_TOL, "\n".join(report)
    print("\n".join(report))
