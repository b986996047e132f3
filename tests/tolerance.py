"""Parity bounds shared by the GPU tests.

The pass rules, derived from the arithmetic (per output element, with S the
oracle's sum_k |w_k x_k|):

* fp32 output of a matvec: |y - y_ref| <= 2e-3 * S.
* bf16 output: the fp32 result is rounded to nearest-even bf16 once more, which
  moves it by at most 2^-8 of its magnitude (8 significant bits), so the bound
  becomes 2e-3 * S + 2^-8 * (|y_ref| + 2e-3 * S).
* S == 0 (all weights or activations zero): the output must be exactly 0.
* gate+up: out = G(g) u with G = gelu_tanh.  With e_g = 2e-3 S_g and
  e_u = 2e-3 S_u the first-order propagation is |G'(g)| e_g |u| + |G(g)| e_u;
  the second-order terms e_g e_u (|G'(g)| + 1) + 0.5 e_g^2 |u| (|G''| <= 1)
  and 1e-6 |out_ref| (fp32 tanhf and the final products) are added.
* small-M tensor-core tile: 1e-2 * S (bf16 weights and activations, fp32
  accumulation), plus the bf16 output term when the output is bf16.
"""
import numpy as np

BF16_HALF_ULP_REL = 2.0 ** -8


def to_f64(t):
    """torch tensor (fp32 or bf16, any device) -> float64 numpy array."""
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def matvec_bound(y_ref, S, rel=2e-3, out_bf16=False):
    tol = rel * S
    if out_bf16:
        tol = tol + BF16_HALF_ULP_REL * (np.abs(y_ref) + rel * S)
    return tol


def check_matvec(y, y_ref, S, rel=2e-3, out_bf16=False, what=""):
    y = np.asarray(y, dtype=np.float64)
    tol = matvec_bound(y_ref, S, rel, out_bf16)
    zero = S == 0
    assert np.all(y[zero] == 0.0), f"{what}: rows with S == 0 must be exactly 0"
    err = np.abs(y - y_ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {bad.sum()} of {y.size} outside the bound; worst at "
                           f"{int(np.argmax(err - tol))}: y={y.flat[np.argmax(err - tol)]!r} "
                           f"ref={y_ref.flat[np.argmax(err - tol)]!r} S={S.flat[np.argmax(err - tol)]!r}")
    nz = S > 0
    return float((err[nz] / S[nz]).max()) if nz.any() else 0.0


def gateup_bound(ref, oracle, out_bf16=False, rel=2e-3):
    g, u, out, Sg, Su = ref["g"], ref["u"], ref["out"], ref["Sg"], ref["Su"]
    eg, eu = rel * Sg, rel * Su
    G = oracle.gelu_tanh(g)
    dG = np.abs(oracle.gelu_tanh_deriv(g))
    tol = dG * eg * np.abs(u) + np.abs(G) * eu + eg * eu * (dG + 1.0) + 0.5 * eg * eg * np.abs(u) \
        + 1e-6 * np.abs(out)
    if out_bf16:
        tol = tol + BF16_HALF_ULP_REL * (np.abs(out) + tol)
    return tol


def check_gateup(o, ref, oracle, out_bf16=False, what=""):
    o = np.asarray(o, dtype=np.float64)
    tol = gateup_bound(ref, oracle, out_bf16)
    err = np.abs(o - ref["out"])
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} of {o.size} outside the bound"
    return float((err / np.maximum(tol, 1e-300)).max())
