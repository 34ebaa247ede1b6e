"""Pins of the fp64 oracle against facts that the definition and mathematics fix.

CPU only.  The oracle states the frame-wise gated delta rule of the SANA-WM
article ("The Architecture": fixed-size state, decay gate, delta-rule
correction, one latent frame per step).  None of these checks re-types that
recurrence: each compares it with an independently derived fact -- a hand
worked example, the token-level gated delta rule, closed forms, exact delta
writes, linearity, an unrolled product formula, permutation invariance,
split/resume, a contraction bound, and the reverse scan.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    """numpy/torch values -> bf16 torch tensor (values chosen exactly representable)."""
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


def rand_inputs(B, H, F, N, dk, dv, seed, s0_std=0.3):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, F, N, H, dk), generator=g).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((B, F, N, H, dk), generator=g), dim=-1).to(torch.bfloat16)
    v = torch.randn((B, F, N, H, dv), generator=g).to(torch.bfloat16)
    beta = torch.rand((B, F, N, H), generator=g) / N
    alpha = 0.8 + 0.2 * torch.rand((B, F, H), generator=g)
    s0 = torch.randn((B, H, dv, dk), generator=g) * s0_std
    return q, k, v, alpha, beta, s0


def run(q, k, v, alpha, beta, s0, **kw):
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    return oracle.frame_forward(q, k, v, alpha, beta, s0, B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def hadamard(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(n)   # n a power of 4 -> entries are exact dyadic numbers


# ---------------------------------------------------------------- hand example
def test_hand_worked_example():
    d = json.load(open(os.path.join(GOLDEN, "hand_d2.json")))
    shp = (d["B"], d["F"], d["N"], d["H"])
    q = bf16(np.reshape(d["q"], shp + (d["dk"],)))
    k = bf16(np.reshape(d["k"], shp + (d["dk"],)))
    v = bf16(np.reshape(d["v"], shp + (d["dv"],)))
    beta = torch.tensor(np.reshape(d["beta"], shp), dtype=torch.float32)
    alpha = torch.tensor(np.reshape(d["alpha"], (d["B"], d["F"], d["H"])), dtype=torch.float32)
    s0 = torch.tensor(np.reshape(d["state_in"], (1, 1, 2, 2)), dtype=torch.float32)
    r = run(q, k, v, alpha, beta, s0)
    np.testing.assert_array_equal(r["out"].reshape(-1), np.reshape(d["expected_out"], -1))
    np.testing.assert_array_equal(r["state"].reshape(-1), np.reshape(d["expected_state"], -1))


# ------------------------------------------------- N=1 == token-level GDN
def token_level_gdn(q, k, v, alpha, beta, s0):
    """Token-by-token gated delta rule (Yang et al., Gated Delta Networks):
    S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T,  o_t = S_t q_t.
    Written per token with rank-1 updates, no frame structure."""
    T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((T, H, dv))
    S = [s0[h].copy() for h in range(H)]
    for t in range(T):
        for h in range(H):
            kt, vt, qt = k[t, h], v[t, h], q[t, h]
            Sk = S[h] @ kt                        # dv
            S[h] = alpha[t, h] * (S[h] - beta[t, h] * np.outer(Sk, kt)) + beta[t, h] * np.outer(vt, kt)
            out[t, h] = S[h] @ qt
    return out, np.stack(S)


@pytest.mark.parametrize("dk,dv", [(8, 6), (16, 16)])
def test_n1_equals_token_level_gated_delta_rule(dk, dv):
    T, H = 37, 3
    q, k, v, alpha, beta, s0 = rand_inputs(1, H, T, 1, dk, dv, seed=11 + dk)
    beta = torch.rand(beta.shape, generator=torch.Generator().manual_seed(5))  # beta in (0,1)
    r = run(q, k, v, alpha, beta, s0)
    o_ref, s_ref = token_level_gdn(f64(q)[0, :, 0], f64(k)[0, :, 0], f64(v)[0, :, 0],
                                   alpha.double().numpy()[0], beta.double().numpy()[0, :, 0],
                                   s0.double().numpy()[0])
    np.testing.assert_allclose(r["out"][0, :, 0], o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["state"][0], s_ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ beta = 0
def test_beta_zero_closed_form():
    B, H, F, N, dk, dv = 2, 3, 5, 7, 8, 6
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=3)
    beta = torch.zeros_like(beta)
    r = run(q, k, v, alpha, beta, s0, want_states=True)
    a = alpha.double().numpy()
    S0 = s0.double().numpy()
    qq = f64(q)
    for b in range(B):
        for h in range(H):
            for f in range(F):
                decay = np.prod(a[b, :f + 1, h])
                np.testing.assert_allclose(r["states"][b, h, f], decay * S0[b, h], rtol=1e-13)
                # O_f = (prod alpha) Q_f S_0^T  (non-symmetric S_0, dk != dv)
                o = decay * qq[b, f, :, h, :] @ S0[b, h].T
                np.testing.assert_allclose(r["out"][b, f, :, h, :], o, rtol=1e-12, atol=1e-14)


# ------------------------------------------------ exact delta write
def test_single_token_unit_key_writes_value():
    dk, dv = 16, 12
    kvec = hadamard(16)[5]                       # unit norm, exact in bf16
    k = bf16(kvec.reshape(1, 1, 1, 1, dk))
    v = bf16(np.linspace(-2, 2, dv).reshape(1, 1, 1, 1, dv))
    q = bf16(kvec.reshape(1, 1, 1, 1, dk))
    s0 = torch.randn((1, 1, dv, dk), generator=torch.Generator().manual_seed(2))
    alpha = torch.ones((1, 1, 1))
    beta = torch.ones((1, 1, 1, 1))
    r = run(q, k, v, alpha, beta, s0)
    S1 = r["state"][0, 0]
    np.testing.assert_allclose(S1 @ kvec, f64(v).reshape(-1), atol=1e-14)
    # the output of a token whose query is the key reads back the value
    np.testing.assert_allclose(r["out"].reshape(-1), f64(v).reshape(-1), atol=1e-14)


def test_orthonormal_keys_multi_token_write_and_decay():
    dk, dv, N = 16, 8, 5
    Hd = hadamard(16)
    keys = Hd[[0, 3, 6, 9, 12]]
    k = bf16(keys.reshape(1, 1, N, 1, dk))
    vals = np.arange(N * dv, dtype=np.float64).reshape(N, dv) / 8.0 - 2.0
    v = bf16(vals.reshape(1, 1, N, 1, dv))
    q = bf16(Hd[[1, 2, 4, 5, 7]].reshape(1, 1, N, 1, dk))
    s0 = torch.randn((1, 1, dv, dk), generator=torch.Generator().manual_seed(9))
    a = 0.625
    alpha = torch.full((1, 1, 1), a)
    beta = torch.ones((1, 1, N, 1))
    r = run(q, k, v, alpha, beta, s0)
    S1 = r["state"][0, 0]
    for i in range(N):
        np.testing.assert_allclose(S1 @ keys[i], vals[i], atol=1e-13)
    # directions orthogonal to every key keep only the decayed old state
    S0 = s0.double().numpy()[0, 0]
    for u in Hd[[1, 2, 4, 5, 7]]:
        np.testing.assert_allclose(S1 @ u, a * (S0 @ u), atol=1e-13)


def test_alpha_zero_forgets_and_scales_write_by_beta():
    dk, dv, N = 16, 8, 4
    Hd = hadamard(16)
    keys = Hd[[2, 5, 11, 14]]
    k = bf16(np.stack([keys, keys]).reshape(1, 2, N, 1, dk))
    vals = np.arange(2 * N * dv).reshape(2, N, dv) / 16.0
    v = bf16(vals.reshape(1, 2, N, 1, dv))
    q = bf16(np.zeros((1, 2, N, 1, dk)))
    betas = np.array([[0.25, 0.5, 0.75, 1.0], [0.125, 0.375, 0.625, 0.875]])
    beta = torch.tensor(betas.reshape(1, 2, N, 1), dtype=torch.float32)
    alpha = torch.zeros((1, 2, 1))
    s0 = torch.randn((1, 1, dv, dk), generator=torch.Generator().manual_seed(1))
    r = run(q, k, v, alpha, beta, s0, want_states=True)
    for f in range(2):
        Sf = r["states"][0, 0, f]
        for i in range(N):
            np.testing.assert_allclose(Sf @ keys[i], betas[f, i] * vals[f, i], atol=1e-14)


# ------------------------------------------------------------ linearity in V
def test_zero_state_linear_in_v():
    B, H, F, N, dk, dv = 1, 2, 6, 5, 8, 8
    g = torch.Generator().manual_seed(4)
    q, k, _, alpha, beta, _ = rand_inputs(B, H, F, N, dk, dv, seed=6)
    v1 = torch.randint(-8, 8, (B, F, N, H, dv), generator=g).float() / 8
    v2 = torch.randint(-8, 8, (B, F, N, H, dv), generator=g).float() / 8
    c = 2.0
    r1 = run(q, k, v1.to(torch.bfloat16), alpha, beta, None)
    r2 = run(q, k, v2.to(torch.bfloat16), alpha, beta, None)
    r12 = run(q, k, (v1 + c * v2).to(torch.bfloat16), alpha, beta, None)
    np.testing.assert_allclose(r12["state"], r1["state"] + c * r2["state"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r12["out"], r1["out"] + c * r2["out"], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ brute-force unroll
def test_unrolled_product_formula():
    """S_F = (prod alpha) S_0 P_1...P_F + sum_f (prod_{g>f} alpha_g) U_f P_{f+1}...P_F,
    P_f = I - A_f, with A_f, U_f built as matrix products K^T diag(beta) K, V^T diag(beta) K."""
    B, H, F, N, dk, dv = 1, 1, 3, 3, 4, 4
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=21, s0_std=1.0)
    beta = beta * N * 0.9
    r = run(q, k, v, alpha, beta, s0, want_states=True)
    K, V, Q = f64(k)[0, :, :, 0], f64(v)[0, :, :, 0], f64(q)[0, :, :, 0]
    be, a, S0 = beta.double().numpy()[0, :, :, 0], alpha.double().numpy()[0, :, 0], s0.double().numpy()[0, 0]
    P = [np.eye(dk) - K[f].T @ np.diag(be[f]) @ K[f] for f in range(F)]
    Uf = [V[f].T @ np.diag(be[f]) @ K[f] for f in range(F)]
    for last in range(F):
        Sx = np.prod(a[:last + 1]) * S0
        for f in range(last + 1):
            Sx = Sx @ P[f]
        for f in range(last + 1):
            term = np.prod(a[f + 1:last + 1]) * Uf[f]
            for g in range(f + 1, last + 1):
                term = term @ P[g]
            Sx = Sx + term
        np.testing.assert_allclose(r["states"][0, 0, last], Sx, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["out"][0, last, :, 0], Q[last] @ Sx.T, rtol=1e-12, atol=1e-14)


# ------------------------------------------------ within-frame permutation
def test_within_frame_permutation():
    B, H, F, N, dk, dv = 1, 2, 3, 9, 8, 8
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=8)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(0))
    r = run(q, k, v, alpha, beta, s0)
    rp = run(q[:, :, perm], k[:, :, perm], v[:, :, perm], alpha, beta[:, :, perm], s0)
    np.testing.assert_allclose(rp["state"], r["state"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(rp["out"], r["out"][:, :, perm.numpy()], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ split/resume
def test_split_resume():
    B, H, F, N, dk, dv = 2, 2, 7, 6, 8, 8
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=12)
    full = run(q, k, v, alpha, beta, s0)
    F1 = 3
    a = run(q[:, :F1], k[:, :F1], v[:, :F1], alpha[:, :F1], beta[:, :F1], s0)
    mid = torch.tensor(a["state"], dtype=torch.float32)   # state is handed over in fp32
    b = run(q[:, F1:], k[:, F1:], v[:, F1:], alpha[:, F1:], beta[:, F1:], mid)
    np.testing.assert_allclose(a["out"], full["out"][:, :F1], rtol=1e-12, atol=1e-14)
    scale = np.abs(full["state"]).max()
    np.testing.assert_allclose(b["state"], full["state"], atol=1e-6 * scale)
    np.testing.assert_allclose(b["out"], full["out"][:, F1:], atol=1e-6 * np.abs(full["out"]).max())


# -------------------------------------------------------- contraction bound
def test_contraction_bound():
    B, H, F, N, dk, dv = 1, 2, 8, 12, 8, 8
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=13, s0_std=10.0)
    beta = 0.9 * beta / beta.sum(dim=2, keepdim=True)   # sum_n beta = 0.9 per (frame, head)
    v = (v.float() * 0.01).to(torch.bfloat16)
    r = run(q, k, v, alpha, beta, s0, want_states=True)
    K, V = f64(k)[0], f64(v)[0]
    be, a = beta.double().numpy()[0], alpha.double().numpy()[0]
    knorm2 = (K ** 2).sum(-1)
    for h in range(H):
        prev = s0.double().numpy()[0, h]
        for f in range(F):
            assert (be[f, :, h] * knorm2[f, :, h]).sum() <= 1.0
            Uf = np.einsum("n,ni,nj->ij", be[f, :, h], V[f, :, h], K[f, :, h])
            cur = r["states"][0, h, f]
            assert np.linalg.norm(cur) <= a[f, h] * np.linalg.norm(prev) + np.linalg.norm(Uf) + 1e-12
            prev = cur


# ------------------------------------------- internal switches and reverse
def test_nodelta_alpha_one_is_cumulative_linear_attention():
    B, H, F, N, dk, dv = 1, 1, 4, 5, 4, 4
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=14)
    alpha = torch.ones_like(alpha)
    r = run(q, k, v, alpha, beta, s0, want_states=True, mode=oracle.MODE_NODELTA)
    # cumulative linear attention: S_f = S_0 + sum_{g<=f} sum_n beta_n v_n k_n^T, built
    # here as one running sum over all tokens up to the end of frame f
    K = f64(k)[0, :, :, 0].reshape(-1, dk)
    V = f64(v)[0, :, :, 0].reshape(-1, dv)
    be = beta.double().numpy()[0, :, :, 0].reshape(-1)
    for f in range(F):
        upto = (f + 1) * N
        Sx = s0.double().numpy()[0, 0] + (V[:upto] * be[:upto, None]).T @ K[:upto]
        np.testing.assert_allclose(r["states"][0, 0, f], Sx, rtol=1e-12, atol=1e-14)


def test_reverse_scan_equals_forward_on_flipped_frames():
    B, H, F, N, dk, dv = 2, 2, 5, 4, 8, 8
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=15)
    rr = run(q, k, v, alpha, beta, s0, mode=oracle.MODE_REVERSE)
    fl = run(q.flip(1), k.flip(1), v.flip(1), alpha.flip(1), beta.flip(1), s0)
    np.testing.assert_allclose(rr["state"], fl["state"], rtol=1e-13, atol=0)
    np.testing.assert_allclose(rr["out"], fl["out"][:, ::-1], rtol=1e-13, atol=0)


# ---------------------------------------------------------- sampling API
def test_sampled_outputs_match_full_outputs():
    w = inputs.WORKLOADS["tiny"]
    x = inputs.workload_inputs(w)
    full = oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"],
                                B=w.B, H=w.H, F=w.F, N=w.N, dk=w.dk, dv=w.dv)
    toks = np.array([0, 5, 17, 63, 40])
    s = oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"],
                             B=w.B, H=w.H, F=w.F, N=w.N, dk=w.dk, dv=w.dv,
                             want_out=False, sample_tokens=toks)
    flat = full["out"].reshape(-1, w.H, w.dv)
    np.testing.assert_array_equal(s["sample_out"], flat[toks])
    np.testing.assert_array_equal(s["state"], full["state"])


def test_oracle_rejects_bad_arguments():
    w = inputs.WORKLOADS["tiny"]
    x = inputs.workload_inputs(w)
    with pytest.raises(RuntimeError):
        oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], None,
                             B=w.B, H=w.H, F=w.F, N=w.N, dk=w.dk, dv=w.dv,
                             want_out=False, sample_tokens=np.array([10 ** 9]))


# ------------------------------------------------ folded prologue (gated entry)
def test_prologue_definition_pins():
    g = torch.Generator().manual_seed(31)
    q = (torch.randn((1, 3, 5, 2, 16), generator=g) * 3).to(torch.bfloat16)
    k = (torch.randn((1, 3, 5, 2, 16), generator=g) * 0.2).to(torch.bfloat16)
    a = torch.tensor([[[-30.0, 0.0], [1.0, 40.0], [-1.0, 2.0]]])
    b = torch.tensor([0.0, 2.0, -2.0, 50.0, -50.0]).repeat(1, 3, 2, 1).permute(0, 1, 3, 2).contiguous()
    qn, kn, alpha, beta = oracle.prologue(q, k, a, b, 0.05)
    np.testing.assert_allclose(np.linalg.norm(qn, axis=-1), 1.0, atol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(kn, axis=-1), 1.0, atol=1e-14)
    # sigmoid fixed points: sigma(0) = 1/2, sigma(2) + sigma(-2) = 1, tails
    assert beta[0, 0, 0, 0] == 0.5
    np.testing.assert_allclose(beta[0, 0, 1, 0] + beta[0, 0, 2, 0], 1.0, atol=1e-15)
    np.testing.assert_allclose(beta[0, 0, 1, 0], 1 / (1 + np.exp(-2.0)), rtol=1e-15)
    assert beta[0, 0, 3, 0] == 1.0 and 0 < beta[0, 0, 4, 0] < 1e-21   # sigma(50) rounds to 1 in fp64
    # softplus(0) = ln 2; softplus(x) ~ x for large x, ~ exp(x) for very negative x
    np.testing.assert_allclose(alpha[0, 0, 1], np.exp(-np.log(2.0) * 0.05), rtol=1e-15)
    np.testing.assert_allclose(alpha[0, 1, 1], np.exp(-40.0 * 0.05), rtol=1e-12)
    np.testing.assert_allclose(alpha[0, 0, 0], np.exp(-np.exp(-30.0) * 0.05), rtol=1e-15)
    # positive rescaling of raw q, k does not change the normalized values
    qn2, kn2, _, _ = oracle.prologue((q.float() * 4).to(torch.bfloat16), (k.float() * 0.5).to(torch.bfloat16),
                                     a, b, 0.05)
    np.testing.assert_allclose(qn2, qn, atol=1e-15)
    np.testing.assert_allclose(kn2, kn, atol=1e-15)


def test_f64_entry_equals_bf16_entry():
    B, H, F, N, dk, dv = 2, 2, 4, 6, 8, 8
    q, k, v, alpha, beta, s0 = rand_inputs(B, H, F, N, dk, dv, seed=41)
    r16 = run(q, k, v, alpha, beta, s0)
    r64 = oracle.frame_forward_f64(f64(q), f64(k), f64(v), alpha.double().numpy(), beta.double().numpy(),
                                   s0.double().numpy(), B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    np.testing.assert_array_equal(r64["out"], r16["out"])
    np.testing.assert_array_equal(r64["state"], r16["state"])


def test_e4m3_decoder_pins():
    """The oracle's e4m3 decoder against values the OCP FP8 format fixes, and
    against torch's own float8_e4m3fn conversion for all 256 codes."""
    spot = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
            0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    codes = np.array(list(spot), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.decode_e4m3(codes), np.array(list(spot.values())))
    assert np.isnan(oracle.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    every = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(every.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(every)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    # positive codes increase strictly; the sign bit only flips the sign
    pos = got[:0x7F]
    assert (np.diff(pos) > 0).all()
    np.testing.assert_array_equal(got[0x80:0xFF], -got[:0x7F])


def test_fp8_forward_equals_bf16_forward_on_shared_values():
    """Every e4m3 value times a power-of-two scale is a bf16 value, so the fp8
    entry (e4m3 decoder) and the bf16 entry (bf16 decoder) see the same
    numbers and must agree exactly."""
    B, H, F, N, dk, dv = 1, 2, 3, 7, 16, 16
    g = torch.Generator().manual_seed(77)
    q8 = torch.randint(0, 0x7F, (B, F, N, H, dk), generator=g, dtype=torch.uint8) | \
        (torch.randint(0, 2, (B, F, N, H, dk), generator=g, dtype=torch.uint8) << 7)
    k8 = torch.randint(0x20, 0x50, (B, F, N, H, dk), generator=g, dtype=torch.uint8)
    v8 = torch.randint(0, 0x7F, (B, F, N, H, dv), generator=g, dtype=torch.uint8)
    sq, sk, sv = 2.0 ** -3, 2.0 ** -6, 0.5
    beta = torch.rand((B, F, N, H), generator=g) / N
    alpha = 0.8 + 0.2 * torch.rand((B, F, H), generator=g)
    s0 = torch.randn((B, H, dv, dk), generator=g) * 0.3
    r8 = oracle.frame_forward_fp8(q8, k8, v8, sq, sk, sv, alpha, beta, s0, B=B, H=H, F=F, N=N, dk=dk, dv=dv)

    def as_bf16(c, s):
        t = c.view(torch.float8_e4m3fn).to(torch.float32) * s
        b = t.to(torch.bfloat16)
        assert torch.equal(b.to(torch.float32), t)  # exactly representable
        return b
    r16 = run(as_bf16(q8, sq), as_bf16(k8, sk), as_bf16(v8, sv), alpha, beta, s0)
    np.testing.assert_array_equal(r8["out"], r16["out"])
    np.testing.assert_array_equal(r8["state"], r16["state"])


def test_e2m1_decoder_pins():
    """The oracle's E2M1 decoder against what a binary floating-point format
    with one sign bit, a 2-bit exponent of bias 1 and a 1-bit mantissa (no
    infinities, no NaN) fixes: exponent field 1 is the binade [1, 2); each
    binade holds two values, the second 1.5 times the first; each next binade
    doubles; the subnormal step equals the first binade's step; the sign bit
    only flips the sign.  Every value is also an exact E4M3 value (torch's
    float8_e4m3fn conversion as the check)."""
    v = oracle.decode_e2m1(np.arange(16))

    def val(e, m):
        return v[(e << 1) | m]
    assert val(0, 0) == 0.0 and val(1, 0) == 1.0
    for e in (1, 2, 3):
        assert val(e, 1) == 1.5 * val(e, 0)
    for e in (1, 2):
        assert val(e + 1, 0) == 2.0 * val(e, 0)
    assert val(0, 1) - val(0, 0) == (val(1, 1) - val(1, 0))
    assert val(3, 1) == 6.0                       # (2 - 2^-1) * 2^(3 - 1): the largest magnitude
    assert (np.diff(v[:8]) > 0).all()
    np.testing.assert_array_equal(v[8:], -v[:8])
    as_e4m3 = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(as_e4m3, v)


def test_nvfp4_layout_worked_example():
    """A hand-decoded 32-element row: nibble order (element 2i low, 2i+1 high),
    one E4M3 scale per 16 elements, the tensor scale on top."""
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0] = 0x21          # element 0: code 1 (0.5), element 1: code 2 (1.0)
    packed[0, 7] = 0xF7          # element 14: code 7 (6.0), element 15: code 15 (-6.0)
    packed[0, 8] = 0x9B          # element 16: code 11 (-1.5), element 17: code 9 (-0.5)
    scales = np.array([[0x40, 0x30]], dtype=np.uint8)   # e4m3 2.0 for elements 0-15, 0.5 for 16-31
    x = oracle.decode_nvfp4(packed, scales, 3.0)
    want = np.zeros((1, 32))
    want[0, 0], want[0, 1] = 0.5 * 2.0 * 3.0, 1.0 * 2.0 * 3.0
    want[0, 14], want[0, 15] = 6.0 * 2.0 * 3.0, -6.0 * 2.0 * 3.0
    want[0, 16], want[0, 17] = -1.5 * 0.5 * 3.0, -0.5 * 0.5 * 3.0
    np.testing.assert_array_equal(x, want)


def test_nvfp4_quantizer_picks_the_nearest_value():
    """Brute force over all 15 E2M1 values of each element's block: the input
    generator's codes are nearest to x / (tensor scale * block scale)."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn((4, 3, 64), generator=g) * torch.tensor([0.01, 1.0, 30.0]).view(1, 3, 1)
    packed, sc, gs = inputs.quantize_nvfp4(x)
    xd = oracle.decode_nvfp4(packed, sc, gs)
    s = np.repeat(oracle.decode_e4m3(sc.numpy()), 16, axis=-1) * gs
    cand = oracle.decode_e2m1(np.arange(16))[None, None, None, :] * s[..., None]   # [..., 64, 16]
    best = np.abs(cand - x.double().numpy()[..., None]).min(axis=-1)
    np.testing.assert_allclose(np.abs(xd - x.double().numpy()), best, rtol=0, atol=1e-12)
    # the block scale never clips: every |x| fits under 6 * block scale (to E4M3 rounding)
    assert (np.abs(x.double().numpy()) <= 6.0 * s * (1 + 2.0 ** -3) + 1e-30).all()


def test_nvfp4_forward_is_the_f64_forward_on_decoded_values():
    B, H, F, N, dk, dv = 1, 2, 2, 5, 16, 32
    x = inputs.draw_nvfp4(B, H, F, N, dk, dv, seed=9, s0_std=0.1)
    r4 = oracle.frame_forward_nvfp4(x["q4"], x["k4"], x["v4"], x["q_sf"], x["k_sf"], x["v_sf"],
                                    x["q_gs"], x["k_gs"], x["v_gs"], x["alpha"], x["beta"], x["state_in"],
                                    B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    dec = {n: oracle.decode_nvfp4(x[n + "4"], x[n + "_sf"], x[n + "_gs"]) for n in ("q", "k", "v")}
    r64 = oracle.frame_forward_f64(dec["q"], dec["k"], dec["v"], x["alpha"].double().numpy(),
                                   x["beta"].double().numpy(), x["state_in"].double().numpy(),
                                   B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    np.testing.assert_array_equal(r4["out"], r64["out"])
    np.testing.assert_array_equal(r4["state"], r64["state"])
    assert dec["k"].shape == (B, F, N, H, dk) and dec["v"].shape == (B, F, N, H, dv)


def _f64_problem(B, H, F, N, dk, dv, seed):
    g = np.random.default_rng(seed)
    x = {"q": g.standard_normal((B, F, N, H, dk)), "k": g.standard_normal((B, F, N, H, dk)) * 0.5,
         "v": g.standard_normal((B, F, N, H, dv)), "alpha": 0.6 + 0.4 * g.random((B, F, H)),
         "beta": g.random((B, F, N, H)) / N, "state_in": g.standard_normal((B, H, dv, dk)) * 0.3}
    w = {"d_out": g.standard_normal((B, F, N, H, dv)), "d_state_out": g.standard_normal((B, H, dv, dk))}
    return x, w


def _loss(x, w, dims):
    r = oracle.frame_forward_f64(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], **dims)
    return float((r["out"] * w["d_out"]).sum() + (r["state"] * w["d_state_out"]).sum())


def test_backward_matches_central_differences():
    """Every gradient of the backward oracle against central differences of
    the forward oracle, along random directions (L = <W_o, O> + <W_s, S_F>)."""
    B, H, F, N, dk, dv = 1, 2, 3, 4, 3, 2
    dims = dict(B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    x, w = _f64_problem(B, H, F, N, dk, dv, seed=5)
    gr = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], w["d_out"],
                               w["d_state_out"], **dims)
    names = {"q": "dq", "k": "dk", "v": "dv", "alpha": "d_alpha", "beta": "d_beta", "state_in": "d_state_in"}
    rng = np.random.default_rng(9)
    eps = 1e-6
    for name, gname in names.items():
        for _ in range(3):
            d = rng.standard_normal(x[name].shape)
            xp = dict(x); xp[name] = x[name] + eps * d
            xm = dict(x); xm[name] = x[name] - eps * d
            fd = (_loss(xp, w, dims) - _loss(xm, w, dims)) / (2 * eps)
            an = float((gr[gname] * d).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def _torch_forward(q, k, v, alpha, beta, s0):
    """The forward written as torch operations, differentiated by autograd."""
    B, F, N, H, dk = q.shape
    outs, states = [], []
    for b in range(B):
        ob, sb = [], []
        for h in range(H):
            S = s0[b, h]
            frames = []
            for f in range(F):
                K, V, Q = k[b, f, :, h], v[b, f, :, h], q[b, f, :, h]
                bt = beta[b, f, :, h]
                A = (K * bt[:, None]).T @ K
                U = (V * bt[:, None]).T @ K
                S = alpha[b, f, h] * (S - S @ A) + U
                frames.append(Q @ S.T)
            ob.append(torch.stack(frames))
            sb.append(S)
        outs.append(torch.stack(ob, dim=2))
        states.append(torch.stack(sb))
    return torch.stack(outs), torch.stack(states)


def test_backward_matches_autograd():
    B, H, F, N, dk, dv = 2, 2, 3, 5, 4, 3
    x, w = _f64_problem(B, H, F, N, dk, dv, seed=6)
    t = {n: torch.tensor(a, requires_grad=True) for n, a in x.items()}
    out, st = _torch_forward(t["q"], t["k"], t["v"], t["alpha"], t["beta"], t["state_in"])
    loss = (out * torch.tensor(w["d_out"])).sum() + (st * torch.tensor(w["d_state_out"])).sum()
    loss.backward()
    gr = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], w["d_out"],
                               w["d_state_out"], B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("alpha", "d_alpha"), ("beta", "d_beta"),
                        ("state_in", "d_state_in")):
        np.testing.assert_allclose(gr[gname], t[name].grad.numpy(), rtol=1e-10, atol=1e-12, err_msg=name)


def test_backward_special_cases():
    """alpha = 0 cuts the chain: nothing flows back to S_0, and with no
    upstream state gradient the last frame's beta gradient only sees the
    outputs.  A zero d_state_out equals passing None."""
    B, H, F, N, dk, dv = 1, 1, 2, 3, 3, 3
    dims = dict(B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    x, w = _f64_problem(B, H, F, N, dk, dv, seed=7)
    x["alpha"][:] = 0.0
    gr = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], w["d_out"], None,
                               **dims)
    assert np.all(gr["d_state_in"] == 0.0)
    gz = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], w["d_out"],
                               np.zeros((B, H, dv, dk)), **dims)
    for n in gr:
        np.testing.assert_array_equal(gr[n], gz[n])
