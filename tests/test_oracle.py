"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one step (or the whole stack) against a closed form, an
invariant, a special case or a brute-force scalar re-derivation written
independently here (plain Python loops, ``math``/``cmath``, explicit index
sums), so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.
"""

import cmath
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers

def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _micro_layer(rng, d, H, Hkv, hd, F):
    qw, kvw = H * hd, Hkv * hd
    return {
        "attn_norm": 1.0 + 0.1 * _rand(rng, d),
        "ffn_norm": 1.0 + 0.1 * _rand(rng, d),
        "wq": _rand(rng, qw, d) / math.sqrt(d),
        "wk": _rand(rng, kvw, d) / math.sqrt(d),
        "wv": _rand(rng, kvw, d) / math.sqrt(d),
        "wo": _rand(rng, d, qw) / math.sqrt(qw),
        "w_gate": _rand(rng, F, d) / math.sqrt(d),
        "w_up": _rand(rng, F, d) / math.sqrt(d),
        "w_down": _rand(rng, d, F) / math.sqrt(F),
    }


def _run_layer(x, w, kp, vp, s, H, Hkv, hd, theta=1.0e4, eps=1e-5):
    return oracle.decoder_layer(x, w, kp, vp, s, H, Hkv, hd, theta, eps)


# ------------------------------------------- brute-force scalar restatement

def _bf_matvec(W, vec):
    # y[o] = sum_i W[o][i] * vec[i]   (weights are [out, in])
    return [sum(W[o][i] * vec[i] for i in range(len(vec))) for o in range(len(W))]


def _bf_rms(vec, g, eps):
    ms = sum(t * t for t in vec) / len(vec)
    r = 1.0 / math.sqrt(ms + eps)
    return [vec[i] * r * g[i] for i in range(len(vec))]


def _bf_rope_head(head, pos, theta):
    # channel i pairs with channel i + hd/2; the pair is a complex number
    # turned by pos * theta**(-2i/hd)
    hd = len(head)
    half = hd // 2
    out = list(head)
    for i in range(half):
        z = complex(head[i], head[i + half]) * cmath.exp(1j * pos * theta ** (-2.0 * i / hd))
        out[i], out[i + half] = z.real, z.imag
    return out


def _bf_layer(xs, w, kp, vp, s, H, Hkv, hd, theta, eps):
    """One layer, row by row, with nothing vectorised."""
    W = {k: np.asarray(v).tolist() for k, v in w.items()}
    keys = [[list(kp[j][g]) for g in range(Hkv)] for j in range(s)]
    vals = [[list(vp[j][g]) for g in range(Hkv)] for j in range(s)]
    qs, outs, krows, vrows = [], [], [], []
    # projections + RoPE for every new row first (all rows are in one call)
    for b, x in enumerate(xs):
        n = _bf_rms(x, W["attn_norm"], eps)
        q = _bf_matvec(W["wq"], n)
        k = _bf_matvec(W["wk"], n)
        v = _bf_matvec(W["wv"], n)
        qh = [_bf_rope_head(q[h * hd:(h + 1) * hd], s + b, theta) for h in range(H)]
        kh = [_bf_rope_head(k[g * hd:(g + 1) * hd], s + b, theta) for g in range(Hkv)]
        vh = [v[g * hd:(g + 1) * hd] for g in range(Hkv)]
        qs.append(qh)
        keys.append(kh)
        vals.append(vh)
        krows.append(kh)
        vrows.append(vh)
    for b, x in enumerate(xs):
        o = []
        for h in range(H):
            g = h * Hkv // H
            sc = [sum(qs[b][h][c] * keys[j][g][c] for c in range(hd)) / math.sqrt(hd)
                  for j in range(s + b + 1)]
            mx = max(sc)
            e = [math.exp(t - mx) for t in sc]
            tot = sum(e)
            o.extend(sum(e[j] / tot * vals[j][g][c] for j in range(len(e))) for c in range(hd))
        att = _bf_matvec(W["wo"], o)
        hrow = [x[i] + att[i] for i in range(len(x))]
        m = _bf_rms(hrow, W["ffn_norm"], eps)
        gt = _bf_matvec(W["w_gate"], m)
        up = _bf_matvec(W["w_up"], m)
        act = [gt[f] / (1.0 + math.exp(-gt[f])) * up[f] for f in range(len(gt))]
        dn = _bf_matvec(W["w_down"], act)
        outs.append([hrow[i] + dn[i] for i in range(len(x))])
    return outs, krows, vrows


@pytest.mark.parametrize("s", [0, 3])
def test_stack_matches_brute_force(s):
    rng = np.random.default_rng(11)
    d, H, Hkv, hd, F, B, L = 8, 4, 2, 4, 12, 3, 2
    theta, eps = 37.0, 1e-5
    layers = [_micro_layer(rng, d, H, Hkv, hd, F) for _ in range(L)]
    pk = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    pv = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    x0 = _rand(rng, B, d)
    got, gk, gv = oracle.prefill_dense_stack(x0, layers, pk, pv, s, H, Hkv, hd, theta, eps)
    xs = x0.tolist()
    for l in range(L):
        xs, kr, vr = _bf_layer(xs, layers[l], pk[l].tolist(), pv[l].tolist(), s, H, Hkv, hd,
                               theta, eps)
        np.testing.assert_allclose(gk[l], np.array(kr), rtol=0, atol=1e-12)
        np.testing.assert_allclose(gv[l], np.array(vr), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got, np.array(xs), rtol=0, atol=1e-11)


# --------------------------------------------------------------- attention

def test_attention_brute_force_per_token():
    rng = np.random.default_rng(1)
    B, s, H, Hkv, hd = 5, 3, 6, 2, 8
    q = _rand(rng, B, H, hd)
    k = _rand(rng, s + B, Hkv, hd)
    v = _rand(rng, s + B, Hkv, hd)
    got = oracle.causal_gqa_attention(q, k, v, s)
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            sc = [float(np.dot(q[b, h], k[j, g])) / math.sqrt(hd) for j in range(s + b + 1)]
            mx = max(sc)
            e = [math.exp(t - mx) for t in sc]
            want = sum(e[j] * v[j, g] for j in range(len(e))) / sum(e)
            np.testing.assert_allclose(got[b, h], want, rtol=0, atol=1e-12)


def test_attention_single_token_no_prefix_is_its_own_value():
    rng = np.random.default_rng(2)
    H, Hkv, hd = 8, 2, 16
    q = _rand(rng, 1, H, hd) * 50.0
    k = _rand(rng, 1, Hkv, hd)
    v = _rand(rng, 1, Hkv, hd)
    got = oracle.causal_gqa_attention(q, k, v, 0)
    for h in range(H):
        assert np.array_equal(got[0, h], v[0, h // (H // Hkv)])


def test_attention_equal_keys_average_visible_values():
    # identical keys -> uniform weights over exactly the visible rows
    rng = np.random.default_rng(3)
    B, s, H, Hkv, hd = 6, 4, 4, 4, 8
    q = _rand(rng, B, H, hd)
    k = np.broadcast_to(_rand(rng, 1, Hkv, hd), (s + B, Hkv, hd)).copy()
    v = _rand(rng, s + B, Hkv, hd)
    got = oracle.causal_gqa_attention(q, k, v, s)
    for b in range(B):
        np.testing.assert_allclose(got[b], v[: s + b + 1].mean(axis=0), rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    rng = np.random.default_rng(4)
    B, s, H, Hkv, hd = 4, 2, 6, 2, 8
    q = _rand(rng, B, H, hd)
    k = _rand(rng, s + B, Hkv, hd)
    v = _rand(rng, s + B, Hkv, hd)
    grp = H // Hkv
    k_mha = np.repeat(k, grp, axis=1)
    v_mha = np.repeat(v, grp, axis=1)
    np.testing.assert_allclose(oracle.causal_gqa_attention(q, k, v, s),
                               oracle.causal_gqa_attention(q, k_mha, v_mha, s), rtol=0, atol=1e-13)


# -------------------------------------------------------------------- RoPE

def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(5)
    t = _rand(rng, 1, 3, 16)
    assert np.array_equal(oracle.rope_neox(t, np.array([0]), 5e5), t)


def test_rope_two_channels_is_complex_rotation_by_position():
    # hd = 2: omega_0 = theta**0 = 1, so position p turns (u, w) by p radians
    for p in (1, 2, 3, 100):
        u, w = 0.3, -1.7
        z = complex(u, w) * cmath.exp(1j * p)
        got = oracle.rope_neox(np.array([[[u, w]]]), np.array([p]), 123.0)[0, 0]
        np.testing.assert_allclose(got, [z.real, z.imag], rtol=0, atol=1e-14)


def test_rope_pairs_channel_i_with_i_plus_half_and_frequency():
    # hd = 4, theta = 100: omega = (1, 0.1).  A vector on channel 1 only
    # turns into channels 1 and 3 by the angle 0.1 * p.
    t = np.zeros((1, 1, 4))
    t[0, 0, 1] = 1.0
    got = oracle.rope_neox(t, np.array([10]), 100.0)[0, 0]
    np.testing.assert_allclose(got, [0.0, math.cos(1.0), 0.0, math.sin(1.0)], rtol=0, atol=1e-14)


def test_rope_preserves_norm_and_is_relative():
    rng = np.random.default_rng(6)
    hd, theta = 64, 5e5
    q = _rand(rng, 1, 1, hd)
    k = _rand(rng, 1, 1, hd)
    for p in (1, 17, 4095):
        qr = oracle.rope_neox(q, np.array([p]), theta)
        assert abs(np.linalg.norm(qr) - np.linalg.norm(q)) < 1e-12
    dots = []
    for m, n in ((9, 4), (109, 104), (2009, 2004)):
        qm = oracle.rope_neox(q, np.array([m]), theta)
        kn = oracle.rope_neox(k, np.array([n]), theta)
        dots.append(float(np.sum(qm * kn)))
    np.testing.assert_allclose(dots, dots[0], rtol=0, atol=1e-11)


# ----------------------------------------------------------------- RMSNorm

def test_rms_norm_hand_value():
    # mean(3^2, 4^2) = 12.5
    got = oracle.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.5)
    np.testing.assert_allclose(got, [[3.0 / math.sqrt(13.0), 8.0 / math.sqrt(13.0)]], rtol=1e-15)


def test_rms_norm_unit_gain_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(7)
    x = _rand(rng, 3, 512)
    y = oracle.rms_norm(x, np.ones(512), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)
    g = 1 + 0.1 * _rand(rng, 512)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, g, 0.0), oracle.rms_norm(x, g, 0.0), rtol=1e-13)


# ------------------------------------------------------------------ SwiGLU

def test_silu_special_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.silu(np.array([60.0])), [60.0], rtol=1e-15)
    assert abs(oracle.silu(np.array([-60.0]))[0]) < 1e-24
    t = np.linspace(-9, 9, 37)
    # t*sigma(t) - (-t)*sigma(-t) = t*(sigma(t)+sigma(-t)) = t
    np.testing.assert_allclose(oracle.silu(t) - oracle.silu(-t), t, rtol=0, atol=1e-14)


# ---------------------------------------------------------- layer / stack

def test_zero_output_projections_make_identity_layer():
    rng = np.random.default_rng(8)
    d, H, Hkv, hd, F, B, s = 16, 4, 2, 4, 24, 5, 3
    w = _micro_layer(rng, d, H, Hkv, hd, F)
    w["wo"] = np.zeros_like(w["wo"])
    w["w_down"] = np.zeros_like(w["w_down"])
    x = _rand(rng, B, d)
    kp, vp = _rand(rng, s, Hkv, hd), _rand(rng, s, Hkv, hd)
    y, k, v = _run_layer(x, w, kp, vp, s, H, Hkv, hd)
    assert np.array_equal(y, x)
    n = oracle.rms_norm(x, w["attn_norm"], 1e-5)
    np.testing.assert_allclose(v, (n @ w["wv"].T).reshape(B, Hkv, hd), rtol=0, atol=1e-14)
    k_direct = oracle.rope_neox((n @ w["wk"].T).reshape(B, Hkv, hd), s + np.arange(B), 1e4)
    np.testing.assert_allclose(k, k_direct, rtol=0, atol=1e-14)


def _stack(x, layers, pk, pv, s, H, Hkv, hd):
    return oracle.prefill_dense_stack(x, layers, pk, pv, s, H, Hkv, hd, 1e4, 1e-5)


def test_decode_equals_prefill():
    rng = np.random.default_rng(9)
    d, H, Hkv, hd, F, B, s, L = 32, 4, 2, 8, 48, 6, 2, 3
    layers = [_micro_layer(rng, d, H, Hkv, hd, F) for _ in range(L)]
    pk = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    pv = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    x = _rand(rng, B, d)
    full, fk, fv = _stack(x, layers, pk, pv, s, H, Hkv, hd)
    ck, cv = [p.copy() for p in pk], [p.copy() for p in pv]
    for b in range(B):
        y, k, v = _stack(x[b:b + 1], layers, ck, cv, s + b, H, Hkv, hd)
        np.testing.assert_allclose(y[0], full[b], rtol=0, atol=1e-12)
        for l in range(L):
            np.testing.assert_allclose(k[l][0], fk[l][b], rtol=0, atol=1e-12)
            np.testing.assert_allclose(v[l][0], fv[l][b], rtol=0, atol=1e-12)
            ck[l] = np.concatenate([ck[l], k[l]], axis=0)
            cv[l] = np.concatenate([cv[l], v[l]], axis=0)


def test_causality_future_row_does_not_change_earlier_rows():
    rng = np.random.default_rng(10)
    d, H, Hkv, hd, F, B, s, L = 32, 4, 2, 8, 48, 7, 3, 2
    layers = [_micro_layer(rng, d, H, Hkv, hd, F) for _ in range(L)]
    pk = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    pv = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    x = _rand(rng, B, d)
    j = 4
    x2 = x.copy()
    x2[j] += 3.0
    a, ak, av = _stack(x, layers, pk, pv, s, H, Hkv, hd)
    b, bk, bv = _stack(x2, layers, pk, pv, s, H, Hkv, hd)
    assert np.array_equal(a[:j], b[:j])
    assert not np.allclose(a[j:], b[j:])
    for l in range(L):
        assert np.array_equal(ak[l][:j], bk[l][:j]) and np.array_equal(av[l][:j], bv[l][:j])


def test_tiny_workload_runs_and_is_finite():
    dims = synth.CONFIGS["tiny"]
    layers, pk, pv, h = synth.draw_workload(dims)
    x, k, v = oracle.prefill_dense_stack(h, layers, pk, pv, dims.start_pos, dims.n_heads,
                                         dims.n_kv_heads, dims.head_dim, dims.rope_theta,
                                         dims.rms_eps)
    assert x.shape == (dims.batch, dims.d_model) and np.all(np.isfinite(x))
    assert len(k) == dims.n_layers and k[0].shape == (dims.batch, dims.n_kv_heads, dims.head_dim)


# ------------------------------------------------------- the pages' figure

def test_host_body_traffic_figure_matches_the_3b_shape():
    """The pages' 111 MB per layer at pp512 follows from the 3B shape's dims."""
    fx = json.load(open(os.path.join(GOLDEN, "host_body_traffic.json")))
    dm = synth.CONFIGS["llama3.2-3b-pp512"]
    assert dm.batch == fx["batch"]
    d, qw, kvw, f = dm.d_model, dm.q_width, dm.kv_width, dm.ffn_dim
    # (in, out) widths of wq, wk, wv, wo, gate, up, down
    mm = [(d, qw), (d, kvw), (d, kvw), (qw, d), (d, f), (d, f), (f, d)]
    assert len(mm) == fx["round_trips"]
    total = sum(dm.batch * (i + o) * 4 for i, o in mm)
    assert round(total / 1e6) == fx["megabytes_decimal"]


# ------------------------------------------------------------ input recipe

def test_bf16_round_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e38],
                    dtype=np.float32)
    want = np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 2.9975342e38], dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.bf16_round(vals))
    np.testing.assert_array_equal(got[:5], want[:5])
    assert abs(got[5] - 3.0e38) / 3.0e38 < 2 ** -8
    np.testing.assert_array_equal(oracle.widen_bf16(synth.bf16_round(vals[:5])), want[:5])


def test_inputs_are_seeded_and_row_stable():
    dims = synth.CONFIGS["tiny"]
    a = synth.draw_hidden(dims)
    b = synth.draw_hidden(dims.replace(batch=3))
    assert np.array_equal(a[:3], b)
    l1 = synth.draw_layer(dims, 1)
    l1b = synth.draw_workload(dims)[0][1]
    for n in synth.LAYER_TENSORS:
        assert np.array_equal(l1[n], l1b[n])
    w = oracle.widen_bf16(l1["w_down"])
    assert abs(w.std() * math.sqrt(dims.ffn_dim) - 1.0) < 0.02


# ------------------------------------------- attention extras and variants
#
# The optional parts of the launch descriptor (cuda_prefill.rs,
# AttnExtrasCuda, LayerRopeCuda, PrefillParams.attn_softcap / window),
# pinned by a second scalar restatement and by closed forms.

def _bf_rope_general(head, pos, theta, layout, rot, ff, mscale):
    # the first `rot` channels form rot/2 complex numbers, each turned by
    # pos * theta**(-2i/rot) / ff[i] and scaled by mscale; the rest stay
    out = list(head)
    half = rot // 2
    for i in range(half):
        a, b = (i, i + half) if layout == "neox" else (2 * i, 2 * i + 1)
        omega = theta ** (-2.0 * i / rot) / (ff[i] if ff is not None else 1.0)
        z = complex(head[a], head[b]) * mscale * cmath.exp(1j * pos * omega)
        out[a], out[b] = z.real, z.imag
    return out


def _bf_layer_variants(xs, w, kp, vp, s, H, Hkv, hd, theta, eps, layout, rot, ff, mscale,
                       softcap, window):
    W = {k: np.asarray(v).tolist() for k, v in w.items()}
    keys = [[list(kp[j][g]) for g in range(Hkv)] for j in range(s)]
    vals = [[list(vp[j][g]) for g in range(Hkv)] for j in range(s)]
    qs, outs, krows, vrows = [], [], [], []

    def heads(vec, nh, bias, gain, pos, rotate):
        if bias is not None:
            vec = [vec[i] + bias[i] for i in range(len(vec))]
        hs = [vec[h * hd:(h + 1) * hd] for h in range(nh)]
        if gain is not None:
            hs = [_bf_rms(t, gain, eps) for t in hs]
        if rotate:
            hs = [_bf_rope_general(t, pos, theta, layout, rot, ff, mscale) for t in hs]
        return hs

    for b, x in enumerate(xs):
        n = _bf_rms(x, W["attn_norm"], eps)
        qh = heads(_bf_matvec(W["wq"], n), H, W.get("q_bias"), W.get("q_norm"), s + b, True)
        kh = heads(_bf_matvec(W["wk"], n), Hkv, W.get("k_bias"), W.get("k_norm"), s + b, True)
        vh = heads(_bf_matvec(W["wv"], n), Hkv, W.get("v_bias"), None, s + b, False)
        qs.append(qh)
        keys.append(kh)
        vals.append(vh)
        krows.append(kh)
        vrows.append(vh)
    for b, x in enumerate(xs):
        p = s + b
        o = []
        for h in range(H):
            g = h * Hkv // H
            seen = [j for j in range(p + 1) if window is None or p - j < window]
            sc = []
            for j in seen:
                z = sum(qs[b][h][c] * keys[j][g][c] for c in range(hd)) / math.sqrt(hd)
                sc.append(softcap * math.tanh(z / softcap) if softcap is not None else z)
            mx = max(sc)
            e = [math.exp(t - mx) for t in sc]
            tot = sum(e)
            o.extend(sum(e[i] / tot * vals[seen[i]][g][c] for i in range(len(seen)))
                     for c in range(hd))
        att = _bf_matvec(W["wo"], o)
        hrow = [x[i] + att[i] for i in range(len(x))]
        m = _bf_rms(hrow, W["ffn_norm"], eps)
        gt = _bf_matvec(W["w_gate"], m)
        up = _bf_matvec(W["w_up"], m)
        act = [gt[f] / (1.0 + math.exp(-gt[f])) * up[f] for f in range(len(gt))]
        dn = _bf_matvec(W["w_down"], act)
        outs.append([hrow[i] + dn[i] for i in range(len(x))])
    return outs, krows, vrows


VARIANTS = {
    "extras": dict(extras=True),
    "norm-layout": dict(rope_layout="norm"),
    "partial-rot-factors-mscale": dict(rot_dim=4, freq_factors=[1.0, 8.0], rope_mscale=1.3),
    "norm-partial": dict(rope_layout="norm", rot_dim=4, extras=True),
    "softcap-window": dict(attn_softcap=0.9, window=3),
    "everything": dict(extras=True, rope_layout="norm", rot_dim=4, freq_factors=[2.0, 0.5],
                       rope_mscale=0.8, attn_softcap=1.5, window=4),
}


@pytest.mark.parametrize("s", [0, 3])
@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_stack_variants_match_brute_force(name, s):
    opts = dict(VARIANTS[name])
    extras = opts.pop("extras", False)
    rng = np.random.default_rng(23)
    d, H, Hkv, hd, F, B, L = 8, 4, 2, 8, 12, 3, 2
    theta, eps = 37.0, 1e-5
    layers = [_micro_layer(rng, d, H, Hkv, hd, F) for _ in range(L)]
    if extras:
        for w in layers:
            w["q_bias"] = 0.3 * _rand(rng, H * hd)
            w["k_bias"] = 0.3 * _rand(rng, Hkv * hd)
            w["v_bias"] = 0.3 * _rand(rng, Hkv * hd)
            w["q_norm"] = 1.0 + 0.2 * _rand(rng, hd)
            w["k_norm"] = 1.0 + 0.2 * _rand(rng, hd)
    pk = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    pv = [_rand(rng, s, Hkv, hd) for _ in range(L)]
    x0 = _rand(rng, B, d)
    got, gk, gv = oracle.prefill_dense_stack(x0, layers, pk, pv, s, H, Hkv, hd, theta, eps,
                                             **opts)
    bf = dict(layout=opts.get("rope_layout", "neox"), rot=opts.get("rot_dim") or hd,
              ff=opts.get("freq_factors"), mscale=opts.get("rope_mscale", 1.0),
              softcap=opts.get("attn_softcap"), window=opts.get("window"))
    xs = x0.tolist()
    for l in range(L):
        xs, kr, vr = _bf_layer_variants(xs, layers[l], pk[l].tolist(), pv[l].tolist(), s, H,
                                        Hkv, hd, theta, eps, **bf)
        np.testing.assert_allclose(gk[l], np.array(kr), rtol=0, atol=1e-12)
        np.testing.assert_allclose(gv[l], np.array(vr), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got, np.array(xs), rtol=0, atol=1e-11)


def test_norm_layout_is_neox_on_interleaved_channels():
    # moving channel 2i to i and 2i+1 to i + hd/2 turns the Norm layout into Neox
    rng = np.random.default_rng(5)
    hd = 8
    t = _rand(rng, 4, 3, hd)
    pos = np.array([0, 1, 7, 40])
    perm = np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])
    got = oracle.rope_rotate(t, pos, 1e4, layout="norm")
    want = oracle.rope_rotate(t[..., perm], pos, 1e4, layout="neox")
    np.testing.assert_allclose(got[..., perm], want, rtol=0, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.rope_rotate(t, pos, 1e4, layout="bogus")


@pytest.mark.parametrize("layout", ["neox", "norm"])
def test_partial_rotation_leaves_the_tail_and_rotates_the_head_as_a_smaller_rope(layout):
    rng = np.random.default_rng(6)
    hd, rot = 16, 8
    t = _rand(rng, 5, 2, hd)
    pos = np.arange(5) * 3 + 1
    got = oracle.rope_rotate(t, pos, 500.0, layout=layout, rot_dim=rot)
    np.testing.assert_array_equal(got[..., rot:], t[..., rot:])
    np.testing.assert_allclose(got[..., :rot], oracle.rope_rotate(t[..., :rot], pos, 500.0,
                                                                  layout=layout),
                               rtol=0, atol=1e-13)


def test_freq_factors_divide_the_angle_and_mscale_scales_the_rotated_channels():
    rng = np.random.default_rng(7)
    hd = 8
    t = _rand(rng, 3, 2, hd)
    pos = np.array([2.0, 6.0, 10.0])
    c = 4.0
    # a common factor c is the same as positions p / c
    np.testing.assert_allclose(oracle.rope_rotate(t, pos, 1e4, freq_factors=[c] * (hd // 2)),
                               oracle.rope_rotate(t, pos / c, 1e4), rtol=0, atol=1e-13)
    # the angular frequencies themselves
    np.testing.assert_allclose(oracle.rope_inv_freq(8, 100.0, [1, 2, 4, 8]),
                               [1.0, 100 ** -0.25 / 2, 100 ** -0.5 / 4, 100 ** -0.75 / 8])
    # mscale multiplies the norm of every rotated pair
    got = oracle.rope_rotate(t, pos, 1e4, rot_dim=4, mscale=1.7)
    for i in range(2):
        a = np.hypot(got[..., i], got[..., i + 2])
        np.testing.assert_allclose(a, 1.7 * np.hypot(t[..., i], t[..., i + 2]), rtol=1e-13)
    np.testing.assert_array_equal(got[..., 4:], t[..., 4:])


def test_window_of_one_row_returns_the_rows_own_value():
    rng = np.random.default_rng(8)
    B, s, H, Hkv, hd = 4, 5, 4, 2, 8
    q = _rand(rng, B, H, hd)
    k = _rand(rng, s + B, Hkv, hd)
    v = _rand(rng, s + B, Hkv, hd)
    o = oracle.causal_gqa_attention(q, k, v, s, window=1)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(o[b, h], v[s + b, h // 2], rtol=0, atol=1e-14)
    # a window at least as long as every row's history changes nothing
    np.testing.assert_allclose(oracle.causal_gqa_attention(q, k, v, s, window=s + B),
                               oracle.causal_gqa_attention(q, k, v, s), rtol=0, atol=0)


def test_softcap_bounds_the_scores_and_vanishes_for_a_wide_cap():
    rng = np.random.default_rng(9)
    B, s, H, Hkv, hd = 3, 2, 2, 1, 4
    q = 4.0 * _rand(rng, B, H, hd)
    k = 4.0 * _rand(rng, s + B, Hkv, hd)
    v = _rand(rng, s + B, Hkv, hd)
    base = oracle.causal_gqa_attention(q, k, v, s)
    wide = oracle.causal_gqa_attention(q, k, v, s, softcap=1e6)
    np.testing.assert_allclose(wide, base, rtol=0, atol=1e-9)
    # with a cap far below the scores every visible key scores about +-cap:
    # two keys, row 0 at s=0 sees key 0 only, row 1 sees two nearly equal weights
    # when both raw scores are large and positive
    q2 = np.ones((2, 1, 4)) * 10.0
    k2 = np.ones((2, 1, 4)) * np.array([[[3.0]], [[5.0]]])
    v2 = np.array([[[1.0, 0, 0, 0]], [[0, 1.0, 0, 0]]])
    o2 = oracle.causal_gqa_attention(q2, k2, v2, 0, softcap=1e-3)
    np.testing.assert_allclose(o2[1, 0, :2], [0.5, 0.5], atol=1e-6)


def test_biases_and_qk_norm_closed_forms():
    rng = np.random.default_rng(10)
    d, H, Hkv, hd, F, B = 8, 2, 1, 8, 12, 3
    w = _micro_layer(rng, d, H, Hkv, hd, F)
    # zero projections: the K/V rows are the rotated k bias and the v bias
    for n in ("wq", "wk", "wv"):
        w[n] = np.zeros_like(w[n])
    w["q_bias"] = _rand(rng, H * hd)
    w["k_bias"] = _rand(rng, Hkv * hd)
    w["v_bias"] = _rand(rng, Hkv * hd)
    x = _rand(rng, B, d)
    empty = np.zeros((0, Hkv, hd))
    _, k, v = oracle.decoder_layer(x, w, empty, empty, 0, H, Hkv, hd, 1e4, 1e-5)
    pos = np.arange(B)
    np.testing.assert_allclose(v, np.broadcast_to(w["v_bias"].reshape(1, Hkv, hd), v.shape),
                               rtol=0, atol=0)
    want_k = oracle.rope_rotate(np.broadcast_to(w["k_bias"].reshape(1, Hkv, hd), k.shape), pos,
                                1e4)
    np.testing.assert_allclose(k, want_k, rtol=0, atol=1e-14)
    # unit k_norm gain: every rotated k head has RMS 1 (eps aside; RoPE keeps norms)
    w2 = _micro_layer(rng, d, H, Hkv, hd, F)
    w2["k_norm"] = np.ones(hd)
    _, k2, _ = oracle.decoder_layer(x, w2, empty, empty, 0, H, Hkv, hd, 1e4, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(k2 ** 2, axis=-1)), 1.0, rtol=1e-12)
