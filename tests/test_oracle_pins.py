"""Pins of the CPU oracle to facts other than itself.

Every oracle function is held to a closed form, an invariant, a worked
example from tests/golden/ or brute force, chosen so that a dropped term, a
wrong sign or index, or a transposed operand fails at least one check.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import golden

EPS = 1e-6
rng = np.random.default_rng(1234)


def f16(v):
    return np.array([v], np.float16).view(np.uint8)


def q4k_block(d=1.0, dmin=0.0, scale_bytes=None, qs=None):
    b = np.zeros(144, np.uint8)
    b[0:2] = f16(d)
    b[2:4] = f16(dmin)
    b[4:16] = scale_bytes if scale_bytes is not None else 0
    b[16:144] = qs if qs is not None else 0
    return b


def q6k_block(d=1.0, scales=None, ql=None, qh=None):
    b = np.zeros(210, np.uint8)
    b[0:128] = ql if ql is not None else 0
    b[128:192] = qh if qh is not None else 0
    b[192:208] = (np.asarray(scales, np.int8).view(np.uint8) if scales is not None else 0)
    b[208:210] = f16(d)
    return b


# ------------------------------------------------------------------ dequant

def test_block_sizes_and_q6k_row_bytes():
    g = golden("q6k_row_bytes.json")
    t = synth.q6k_tensor(7, 1, g["k"])
    assert t.data.size == g["row_bytes"]
    assert synth.q4k_tensor(7, 1, 256).data.size == 144
    assert synth.q6k_tensor(7, 1, 256).data.size == 210


def test_fp16_decode_special_values():
    for v in [0.0, -0.0, 1.0, -2.5, 65504.0, 6.103515625e-05, 5.960464477539063e-08, 0.019989013671875]:
        bits = int(np.array([v], np.float16).view(np.uint16)[0])
        assert oracle.lib().or_f16(bits) == np.float32(v)
    assert math.isinf(oracle.lib().or_f16(0x7C00))
    assert math.isnan(oracle.lib().or_f16(0x7E00))


def test_all_zero_blocks_dequantize_to_zero():
    assert np.all(oracle.dequant_block(np.zeros(144, np.uint8), oracle.Q4_K) == 0)
    assert np.all(oracle.dequant_block(np.zeros(210, np.uint8), oracle.Q6_K) == 0)


def test_all_max_q4k_block():
    # q = 15, sc = m = 63 everywhere: weight = 63*(15*d - dmin)
    d, dmin = 0.5, 0.25
    b = q4k_block(d, dmin, np.full(12, 0xFF, np.uint8), np.full(128, 0xFF, np.uint8))
    w = oracle.dequant_block(b, oracle.Q4_K)
    assert np.all(w == np.float32(63 * (15 * d - dmin)))


def test_all_max_q6k_block():
    # q = 63, scale = 127: weight = 127*31*d
    d = 0.5
    b = q6k_block(d, np.full(16, 127), np.full(128, 0xFF, np.uint8), np.full(64, 0xFF, np.uint8))
    w = oracle.dequant_block(b, oracle.Q6_K)
    assert np.all(w == np.float32(127 * 31 * d))


def test_q4k_scale_unpacking_worked_example():
    g = golden("q4k_scales_worked.json")
    sb = np.array(g["scale_bytes"], np.uint8)
    for j in range(8):
        assert oracle.q4k_scale_min(sb, j) == (g["sc"][j], g["m"][j])


def test_q4k_scale_unpacking_is_a_bijection():
    # 12 bytes hold exactly sixteen 6-bit fields: distinct byte strings must
    # give distinct (sc, m) sets, and every bit must matter.
    sb = np.zeros(12, np.uint8)
    base = [oracle.q4k_scale_min(sb, j) for j in range(8)]
    assert base == [(0, 0)] * 8
    for byte in range(12):
        for bit in range(8):
            s = sb.copy()
            s[byte] = 1 << bit
            vals = [oracle.q4k_scale_min(s, j) for j in range(8)]
            assert vals != base, (byte, bit)
            assert sum(v != (0, 0) for v in vals) == 1  # one field changes


def test_q4k_nibble_positions():
    g = golden("q4k_nibble_positions.json")
    sb = np.array([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], np.uint8)
    for p in g["probes"]:
        qs = np.zeros(128, np.uint8)
        qs[p["byte"]] = 0x21
        w = oracle.dequant_block(q4k_block(1.0, 0.0, sb, qs), oracle.Q4_K)
        nz = np.nonzero(w)[0].tolist()
        assert nz == sorted([p["low_weight"], p["high_weight"]])
        assert w[p["low_weight"]] == 1.0 and w[p["high_weight"]] == 2.0


def test_q4k_min_term_and_sub_block_scales():
    # sub-block j has sc = j+1, m = 2j+1: constant q = 3 gives d*(j+1)*3 - dmin*(2j+1)
    sc = [j + 1 for j in range(8)]
    mn = [2 * j + 1 for j in range(8)]
    sb = np.zeros(12, np.uint8)
    for j in range(4):
        sb[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        sb[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        sb[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    assert [oracle.q4k_scale_min(sb, j) for j in range(8)] == list(zip(sc, mn))
    d, dmin = 0.125, 0.0625
    w = oracle.dequant_block(q4k_block(d, dmin, sb, np.full(128, 0x33, np.uint8)), oracle.Q4_K)
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == np.float32(d * sc[j] * 3 - dmin * mn[j]))


def test_q6k_positions():
    g = golden("q6k_positions.json")
    for p in g["probes"]:
        ql, qh = np.zeros(128, np.uint8), np.zeros(64, np.uint8)
        (ql if p["field"] == "ql" else qh)[p["byte"]] = p["value"]
        w = oracle.dequant_block(q6k_block(1.0, np.ones(16), ql, qh), oracle.Q6_K)
        expect = np.full(256, -32.0, np.float32)
        expect[p["weight"]] = p["expect"]
        assert np.array_equal(w, expect), p
    for p in g["scale_probes"]:
        sc = np.ones(16)
        sc[p["scale"]] = 2
        w = oracle.dequant_block(q6k_block(1.0, sc), oracle.Q6_K)
        lo, hi = p["weights"]
        idx = np.nonzero(w == -64.0)[0]
        assert idx.min() == lo and idx.max() == hi and idx.size == hi - lo + 1


def test_q6k_negative_scales_and_offset():
    # q = 0 -> q-32 = -32; scale -128 -> weight = d*(-128)*(-32)
    w = oracle.dequant_block(q6k_block(0.25, np.full(16, -128)), oracle.Q6_K)
    assert np.all(w == np.float32(0.25 * 128 * 32))


# --------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("qtype", [oracle.Q4_K, oracle.Q6_K])
def test_gemv_matches_dense_product_within_f32_bound(qtype):
    n, k = 37, 768
    t = (synth.q4k_tensor if qtype == oracle.Q4_K else synth.q6k_tensor)(99, n, k)
    x = rng.standard_normal(k).astype(np.float32)
    W = oracle.dequant(t).astype(np.float64)
    exact = W @ x.astype(np.float64)
    y32, y64 = oracle.gemv(t, x), oracle.gemv_f64(t, x)
    bound = k * np.finfo(np.float32).eps * (np.abs(W) @ np.abs(x.astype(np.float64)))
    assert np.all(np.abs(y32 - exact) <= bound)
    assert np.allclose(y64, exact, rtol=1e-12, atol=1e-9)
    rows = np.array([0, 5, 36], np.int32)
    assert np.array_equal(oracle.gemv_rows(t, x, rows), y32[rows])


def test_gemv_rows_are_row_major_blocks():
    # row r's bytes start at r * (k/256) * 144: zero one row's blocks -> y[r] = 0
    t = synth.q4k_tensor(5, 4, 512)
    t.data[2 * 288:3 * 288] = 0
    y = oracle.gemv(t, np.ones(512, np.float32))
    assert y[2] == 0 and np.all(y[[0, 1, 3]] != 0)


def test_gemv_thread_count_does_not_change_results():
    t = synth.q4k_tensor(3, 64, 1024)
    x = rng.standard_normal(1024).astype(np.float32)
    n0 = oracle.max_threads()
    oracle.set_threads(1)
    a = oracle.gemv(t, x)
    oracle.set_threads(max(2, n0))
    b = oracle.gemv(t, x)
    oracle.set_threads(n0)
    assert np.array_equal(a, b)


# -------------------------------------------------------------- elementwise

def test_scalar_activations_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.softplus(0.0) - math.log(2)) < 1e-7
    assert oracle.softplus(200.0) == 200.0 and oracle.softplus(-200.0) == 0.0
    assert oracle.silu(-200.0) == 0.0 and oracle.silu(100.0) == 100.0
    for x in [-3.0, -0.5, 0.7, 4.0]:
        assert abs(oracle.silu(x) - x / (1 + math.exp(-x))) < 1e-6 * max(1, abs(x))
        assert abs(oracle.softplus(x) - math.log1p(math.exp(x))) < 1e-6


def test_rmsnorm_constant_vector_and_scale_invariance():
    w = rng.standard_normal(64).astype(np.float32)
    c = 3.0
    y = oracle.rmsnorm(np.full(64, c, np.float32), w)
    assert np.allclose(y, c / math.sqrt(c * c + EPS) * w, rtol=1e-6)
    x = rng.standard_normal(64).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x * 1024, w), oracle.rmsnorm(x, w), rtol=1e-5)
    # unit weights: mean square of the output is 1
    y = oracle.rmsnorm(x, np.ones(64, np.float32))
    assert abs(float(np.mean(y.astype(np.float64) ** 2)) - 1.0) < 1e-5


def test_l2norm_heads_unit_norm_and_direction():
    x = rng.standard_normal(3 * 128).astype(np.float32) * 5
    y = oracle.l2norm_heads(x, 128)
    for h in range(3):
        v = y[128 * h:128 * h + 128].astype(np.float64)
        assert abs(np.linalg.norm(v) - 1.0) < 1e-6
        u = x[128 * h:128 * h + 128].astype(np.float64)
        assert abs(float(v @ u) - np.linalg.norm(u)) < 1e-4 * np.linalg.norm(u)


def test_conv_impulse_weight_gives_silu_and_rolls_window():
    C, K = 10, 4
    wconv = np.zeros((C, K), np.float32)
    wconv[:, K - 1] = 1.0
    x = rng.standard_normal(C).astype(np.float32)
    win = rng.standard_normal((C, K - 1)).astype(np.float32)
    out, win2 = oracle.conv1d_silu(x, win, wconv)
    assert np.allclose(out, [oracle.silu(float(v)) for v in x], rtol=1e-6)
    assert np.array_equal(win2[:, :K - 2], win[:, 1:]) and np.array_equal(win2[:, K - 2], x)


def test_conv_shift_weight_replays_input_three_steps_later():
    C, K = 6, 4
    wconv = np.zeros((C, K), np.float32)
    wconv[:, 0] = 1.0  # the oldest window entry
    win = np.zeros((C, K - 1), np.float32)
    xs = [rng.standard_normal(C).astype(np.float32) for _ in range(6)]
    outs = []
    for x in xs:
        out, win = oracle.conv1d_silu(x, win, wconv)
        outs.append(out)
    for t in range(3, 6):
        assert np.allclose(outs[t], [oracle.silu(float(v)) for v in xs[t - 3]], rtol=1e-6)


def test_conv_weighted_sum_order_of_taps():
    # weights (1,2,3,4) on window (a,b,c) and input x: a + 2b + 3c + 4x
    wconv = np.array([[1, 2, 3, 4]], np.float32)
    win = np.array([[0.5, -1.0, 0.25]], np.float32)
    out, _ = oracle.conv1d_silu(np.array([0.125], np.float32), win, wconv)
    z = 0.5 - 2.0 + 0.75 + 0.5
    assert abs(out[0] - z / (1 + math.exp(-z))) < 1e-6


def test_gates_closed_forms():
    alpha = np.array([0.0, 100.0, -100.0], np.float32)
    bias = np.zeros(3, np.float32)
    a = np.array([-2.0, -0.5, -1.0], np.float32)
    braw = np.array([0.0, 50.0, -50.0], np.float32)
    dt, be = oracle.gates(alpha, bias, a, braw)
    assert abs(dt[0] - (-2.0 * math.log(2))) < 1e-6
    assert dt[1] == -50.0 and abs(dt[2]) < 1e-40  # softplus(-100) = 3.7e-44
    assert be[0] == 0.5 and be[1] == 1.0 and be[2] < 1e-20
    dt2, _ = oracle.gates(np.array([0.5], np.float32), np.array([0.25], np.float32),
                          np.array([-1.0], np.float32), np.zeros(1, np.float32))
    assert abs(dt2[0] + math.log1p(math.exp(0.75))) < 1e-6  # bias is added before softplus


# ----------------------------------------------------------------- delta rule

def _rand_delta(nk=2, nv=4, dk=16, dv=8):
    q = oracle.l2norm_heads(rng.standard_normal(nk * dk), dk)
    k = oracle.l2norm_heads(rng.standard_normal(nk * dk), dk)
    v = rng.standard_normal(nv * dv).astype(np.float32)
    S = rng.standard_normal((nv, dv, dk)).astype(np.float32)
    return q, k, v, S


def test_delta_rule_worked_2x2():
    g = golden("delta_rule_2x2.json")
    S = np.array(g["state_in"], np.float32).reshape(1, 2, 2)
    o, S2 = oracle.delta_rule(g["q"], g["k"], g["v"], [g["beta"]], [g["dt"]], S, 1, 2, 1, 2)
    assert np.allclose(S2.ravel(), g["state_out"], rtol=2e-6)
    assert np.allclose(o, g["o"], rtol=2e-6)


def test_delta_rule_identity_when_g1_beta0():
    nk, nv, dk, dv = 2, 4, 16, 8
    q, k, v, S = _rand_delta(nk, nv, dk, dv)
    o, S2 = oracle.delta_rule(q, k, v, np.zeros(nv), np.zeros(nv), S, nk, dk, nv, dv)
    assert np.array_equal(S2, S)
    for h in range(nv):
        kh = h % nk
        expect = S[h].astype(np.float64) @ q[kh * dk:(kh + 1) * dk].astype(np.float64) / math.sqrt(dk)
        assert np.allclose(o[h * dv:(h + 1) * dv], expect, rtol=1e-5, atol=1e-6)


def test_delta_rule_from_zero_state_is_rank_one():
    nk, nv, dk, dv = 2, 4, 16, 8
    q, k, v, _ = _rand_delta(nk, nv, dk, dv)
    beta = rng.uniform(0.1, 0.9, nv).astype(np.float32)
    dt = rng.uniform(-2, 0, nv).astype(np.float32)
    o, S2 = oracle.delta_rule(q, k, v, beta, dt, np.zeros((nv, dv, dk), np.float32), nk, dk, nv, dv)
    for h in range(nv):
        kh = h % nk
        kk, qq = k[kh * dk:(kh + 1) * dk], q[kh * dk:(kh + 1) * dk]
        for j in range(dv):
            assert np.allclose(S2[h, j], beta[h] * v[h * dv + j] * kk, rtol=1e-6, atol=1e-7)
            assert abs(o[h * dv + j] - beta[h] * v[h * dv + j] * float(kk @ qq) / math.sqrt(dk)) < 1e-5


def test_delta_rule_zero_decay_resets_state():
    nk, nv, dk, dv = 2, 4, 16, 8
    q, k, v, S = _rand_delta(nk, nv, dk, dv)
    beta = np.full(nv, 0.5, np.float32)
    dt = np.full(nv, -np.inf, np.float32)
    o1, S1 = oracle.delta_rule(q, k, v, beta, dt, S, nk, dk, nv, dv)
    o0, S0 = oracle.delta_rule(q, k, v, beta, dt, np.zeros_like(S), nk, dk, nv, dv)
    assert np.array_equal(S1, S0) and np.array_equal(o1, o0)


def test_delta_rule_value_head_uses_key_head_h_mod_nk():
    nk, nv, dk, dv = 2, 4, 16, 8
    q, k, v, S = _rand_delta(nk, nv, dk, dv)
    beta, dt = np.full(nv, 0.7, np.float32), np.full(nv, -0.3, np.float32)
    o, S2 = oracle.delta_rule(q, k, v, beta, dt, S, nk, dk, nv, dv)
    # perturbing key head 1 changes value heads 1 and 3 only
    k2 = k.copy()
    k2[dk:] = oracle.l2norm_heads(rng.standard_normal(dk), dk)
    o2, _ = oracle.delta_rule(q, k2, v, beta, dt, S, nk, dk, nv, dv)
    changed = [h for h in range(nv) if not np.array_equal(o[h * dv:(h + 1) * dv], o2[h * dv:(h + 1) * dv])]
    assert changed == [1, 3]


def test_delta_rule_brute_force_float64():
    nk, nv, dk, dv = 2, 4, 16, 8
    q, k, v, S = _rand_delta(nk, nv, dk, dv)
    beta = rng.uniform(0, 1, nv).astype(np.float32)
    dt = rng.uniform(-1, 0, nv).astype(np.float32)
    o, S2 = oracle.delta_rule(q, k, v, beta, dt, S, nk, dk, nv, dv)
    # matrix form: S_h^T (dk x dv) = g*S^T + k (beta*(v - (g S^T)^T k))^T, o = S_h'^T-columns . q
    for h in range(nv):
        kh = h % nk
        kk = k[kh * dk:(kh + 1) * dk].astype(np.float64)
        qq = q[kh * dk:(kh + 1) * dk].astype(np.float64)
        M = S[h].astype(np.float64).T * math.exp(float(dt[h]))  # M[i, j] = g*S[i][j]
        dvec = float(beta[h]) * (v[h * dv:(h + 1) * dv] - M.T @ kk)
        M2 = M + np.outer(kk, dvec)
        assert np.allclose(S2[h].T, M2, rtol=1e-5, atol=1e-5)
        assert np.allclose(o[h * dv:(h + 1) * dv], M2.T @ qq / math.sqrt(dk), rtol=1e-4, atol=1e-5)


# ----------------------------------------------------------- gated norm, FFN

def test_gated_rmsnorm_closed_forms():
    dv, nv = 8, 3
    w = rng.standard_normal(dv).astype(np.float32)
    o = np.repeat(np.array([2.0, -1.0, 0.5], np.float32), dv)
    z = np.concatenate([np.zeros(dv), np.full(dv, 30.0), np.full(dv, -30.0)]).astype(np.float32)
    u = oracle.gated_rmsnorm(o, z, w, dv)
    assert np.all(u[:dv] == 0)  # silu(0) = 0
    assert np.allclose(u[dv:2 * dv], -1.0 / math.sqrt(1 + EPS) * w * 30.0, rtol=1e-6)
    assert np.allclose(u[2 * dv:], 0.0, atol=1e-10)  # silu(-30) ~ -2.8e-12
    # each head is normalized on its own
    o2 = o.copy()
    o2[:dv] *= 100
    u2 = oracle.gated_rmsnorm(o2, np.ones(nv * dv, np.float32), w, dv)
    u1 = oracle.gated_rmsnorm(o, np.ones(nv * dv, np.float32), w, dv)
    assert np.allclose(u2, u1, rtol=1e-5)


def test_swiglu_closed_form():
    g = np.array([0.0, 1.0, -40.0, 3.0], np.float32)
    up = np.array([5.0, 2.0, 7.0, -1.0], np.float32)
    act = oracle.swiglu(g, up)
    assert act[0] == 0 and abs(act[2]) < 1e-14
    assert abs(act[1] - 2.0 / (1 + math.exp(-1))) < 1e-6
    assert abs(act[3] + 3.0 / (1 + math.exp(-3))) < 1e-6


# ------------------------------------------------------------ attention ops

def test_split_q_gate_brute_force():
    nh, hd = 3, 4
    qf = np.arange(nh * 2 * hd, dtype=np.float32)
    q, gate = oracle.split_q_gate(qf, nh, hd)
    for h in range(nh):
        assert np.array_equal(q[h * hd:(h + 1) * hd], qf[h * 2 * hd:h * 2 * hd + hd])
        assert np.array_equal(gate[h * hd:(h + 1) * hd], qf[h * 2 * hd + hd:(h + 1) * 2 * hd])


def test_rmsnorm_heads_equals_per_slice_rmsnorm():
    x = rng.standard_normal(3 * 16).astype(np.float32)
    w = rng.standard_normal(16).astype(np.float32)
    y = oracle.rmsnorm_heads(x, w, 16)
    for h in range(3):
        assert np.array_equal(y[16 * h:16 * h + 16], oracle.rmsnorm(x[16 * h:16 * h + 16], w))


def test_rope_identity_at_pos0_norm_preserved_tail_untouched():
    hd, n_rot = 32, 8
    ts = oracle.theta_scale(1.0e7, n_rot)
    assert abs(ts - 1.0e7 ** (-2 / n_rot)) < 1e-9
    x = rng.standard_normal(2 * hd).astype(np.float32)
    assert np.array_equal(oracle.rope_neox(x, hd, n_rot, 0, ts), x)
    y = oracle.rope_neox(x, hd, n_rot, 777, ts)
    for h in range(2):
        v, u = x[h * hd:(h + 1) * hd], y[h * hd:(h + 1) * hd]
        assert np.array_equal(u[n_rot:], v[n_rot:])
        for i in range(n_rot // 2):
            a = math.hypot(v[i], v[i + n_rot // 2])
            b = math.hypot(u[i], u[i + n_rot // 2])
            assert abs(a - b) < 1e-5 * max(1, a)


def test_rope_rotation_angles_closed_form():
    hd, n_rot, pos = 16, 8, 5
    ts = 0.5
    half = n_rot // 2
    for i in range(half):
        x = np.zeros(hd, np.float32)
        x[i] = 1.0  # unit vector in the first slot of pair i
        y = oracle.rope_neox(x, hd, n_rot, pos, ts)
        theta = pos * ts ** i
        assert abs(y[i] - math.cos(theta)) < 1e-6 and abs(y[i + half] - math.sin(theta)) < 1e-6
        x2 = np.zeros(hd, np.float32)
        x2[i + half] = 1.0  # second slot rotates to (-sin, cos)
        y2 = oracle.rope_neox(x2, hd, n_rot, pos, ts)
        assert abs(y2[i] + math.sin(theta)) < 1e-6 and abs(y2[i + half] - math.cos(theta)) < 1e-6


def _kv(t, nkv, hd):
    return (rng.standard_normal((t, nkv * hd)).astype(np.float32),
            rng.standard_normal((t, nkv * hd)).astype(np.float32))


def test_attention_single_key_returns_value_row_of_group():
    nh, nkv, hd = 4, 2, 8
    kc, vc = _kv(1, nkv, hd)
    out = oracle.attention(rng.standard_normal(nh * hd), kc, vc, nh, nkv, hd, 1)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.allclose(out[h * hd:(h + 1) * hd], vc[0, g * hd:(g + 1) * hd], rtol=1e-6)


def test_attention_identical_keys_average_values():
    nh, nkv, hd, t = 2, 1, 8, 5
    kc, vc = _kv(t, nkv, hd)
    kc[:] = kc[0]
    out = oracle.attention(rng.standard_normal(nh * hd), kc, vc, nh, nkv, hd, t)
    assert np.allclose(out[:hd], vc.mean(axis=0), rtol=1e-5, atol=1e-6)


def test_attention_two_keys_softmax_closed_form():
    nh, nkv, hd = 1, 1, 4
    q = np.array([1.0, 0, 0, 0], np.float32)
    kc = np.array([[2.0, 0, 0, 0], [0.0, 0, 0, 0]], np.float32)
    vc = np.array([[1.0, 0, 0, 0], [0.0, 1, 0, 0]], np.float32)
    out = oracle.attention(q, kc, vc, nh, nkv, hd, 2)
    s0 = 2.0 / math.sqrt(hd)
    p0 = math.exp(s0) / (math.exp(s0) + 1.0)
    assert np.allclose(out, [p0, 1 - p0, 0, 0], rtol=1e-6, atol=1e-7)
    # rows past t_len are ignored
    kc3 = np.vstack([kc, [[50.0, 0, 0, 0]]]).astype(np.float32)
    vc3 = np.vstack([vc, [[0, 0, 9.0, 0]]]).astype(np.float32)
    assert np.array_equal(oracle.attention(q, kc3, vc3, nh, nkv, hd, 2), out)


def test_sigmoid_gate_closed_form():
    x = np.array([2.0, -4.0, 1.0], np.float32)
    g = np.array([0.0, 100.0, -100.0], np.float32)
    assert np.allclose(oracle.sigmoid_gate(x, g), [1.0, -4.0, 0.0], atol=1e-30)


# ------------------------------------------------------------------- argmax

def test_argmax_first_index_on_planted_ties():
    for trial in range(20):
        x = rng.standard_normal(5000).astype(np.float32)
        idx = np.sort(rng.choice(5000, size=rng.integers(2, 9), replace=False))
        x[idx] = x.max() + 1.0
        assert oracle.argmax(x) == idx[0]


def test_argmax_inf_nan_and_signed_zero():
    x = np.zeros(10, np.float32)
    x[7] = np.inf
    x[3] = np.nan
    assert oracle.argmax(x) == 7
    assert oracle.argmax(np.full(4, np.nan, np.float32)) == 0
    y = np.array([-1.0, -0.0, 0.0, -2.0], np.float32)
    assert oracle.argmax(y) == 1  # -0 == +0: the first wins
    a, b = oracle.top2(np.array([1.0, 5.0, 3.0, 5.0], np.float32))
    assert (a, b) == (5.0, 5.0)


def _allow(n, allowed):
    """Packed allow bitset of n tokens with exactly the ids in `allowed` set."""
    w = np.zeros((n + 31) // 32, np.uint32)
    for i in allowed:
        w[i >> 5] |= np.uint32(1) << np.uint32(i & 31)
    return w


def test_masked_argmax_hand_cases():
    """The grammar mask: banned logits become -FLT_MAX before the first-index
    argmax (values worked by hand)."""
    x = np.array([3.0, 1.0, 3.0, 2.0], np.float32)
    assert oracle.argmax_masked(x, _allow(4, range(4))) == 0   # no ban: first of the tied maxima
    assert oracle.argmax_masked(x, _allow(4, [1, 2, 3])) == 2  # the first maximum banned
    assert oracle.argmax_masked(x, _allow(4, [1, 3])) == 3     # both maxima banned
    assert oracle.argmax_masked(x, _allow(4, [1])) == 1        # one token allowed
    assert oracle.argmax_masked(x, _allow(4, [])) == 0         # all banned: all -FLT_MAX, first index
    # -FLT_MAX (a banned id) is above -inf: an allowed -inf logit loses to the first banned id
    assert oracle.argmax_masked(np.array([5.0, -np.inf], np.float32), _allow(2, [1])) == 0
    # an allowed NaN never wins; ids beyond n in the last word are ignored
    y = np.full(40, -1.0, np.float32)
    y[33], y[38] = np.nan, 0.5
    assert oracle.argmax_masked(y, _allow(40, [33, 38])) == 38
    assert oracle.argmax_masked(y, _allow(40, [33, 38]) | np.array([0, 0xFFFFFF00], np.uint32)) == 38


def test_masked_argmax_equals_argmax_over_allowed_ids():
    """On finite logits the mask is the argmax over the allowed ids alone
    (brute force on random cases)."""
    rng = np.random.default_rng(71)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        x = rng.standard_normal(n).astype(np.float32)
        keep = np.flatnonzero(rng.random(n) < 0.3)
        if keep.size == 0:
            continue
        want = keep[np.argmax(x[keep])]  # numpy's argmax is first-index too
        assert oracle.argmax_masked(x, _allow(n, keep)) == want


# ---------------------------------------------------- layers and whole token

def _zero(t):
    t.data[:] = 0
    return t


def test_deltanet_layer_with_zero_output_projections_leaves_hidden():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    _zero(w.layers[0].ssm_out)
    _zero(w.layers[0].ffn_down)
    m = oracle.Model(w)
    st = oracle.State(m)
    conv0, ssm0 = synth.initial_deltanet_state(cfg, 0)
    st.conv[0][:] = conv0
    st.ssm[0][:] = ssm0
    h = rng.standard_normal(cfg.hidden).astype(np.float32)
    assert np.array_equal(oracle.deltanet_layer(m, st, 0, h), h)
    assert not np.array_equal(st.ssm[0], ssm0)  # the state still advanced


def test_deltanet_layer_with_zero_qkv_only_decays_state():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    L = w.layers[0]
    _zero(L.attn_qkv)
    m = oracle.Model(w)
    st = oracle.State(m)
    ssm0 = synth.initial_deltanet_state(cfg, 0)[1]
    st.ssm[0][:] = ssm0
    h = rng.standard_normal(cfg.hidden).astype(np.float32)
    oracle.deltanet_layer(m, st, 0, h)
    # conv input and window are zero -> q = k = v = 0 -> S' = exp(dt) * S
    xn = oracle.rmsnorm(h, L.attn_norm)
    a = -np.exp(L.ssm_a_log.astype(np.float64))
    al, br = oracle.gemv(L.ssm_alpha, xn), oracle.gemv(L.ssm_beta, xn)
    dt = np.array([math.log1p(math.exp(float(al[i] + L.ssm_dt_bias[i]))) if al[i] + L.ssm_dt_bias[i] < 30
                   else float(al[i] + L.ssm_dt_bias[i]) for i in range(cfg.n_v_heads)]) * a
    for hh in range(cfg.n_v_heads):
        assert np.allclose(st.ssm[0][hh], math.exp(dt[hh]) * ssm0[hh], rtol=2e-5, atol=1e-30)


def test_attention_layer_writes_kv_row_at_pos_and_zero_projections_pass_through():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    il = 3
    L = w.layers[il]
    _zero(L.attn_output)
    _zero(L.ffn_down)
    m = oracle.Model(w)
    st = oracle.State(m)
    h = rng.standard_normal(cfg.hidden).astype(np.float32)
    pos = 7
    assert np.array_equal(oracle.attention_layer(m, st, il, h, pos), h)
    xn = oracle.rmsnorm(h, L.attn_norm)
    assert np.array_equal(st.vc[il][pos], oracle.gemv(L.attn_v, xn))
    krow = oracle.rope_neox(oracle.rmsnorm_heads(oracle.gemv(L.attn_k, xn), L.attn_k_norm, cfg.head_dim),
                            cfg.head_dim, cfg.n_rot, pos, oracle.theta_scale(cfg.rope_theta, cfg.n_rot))
    assert np.array_equal(st.kc[il][pos], krow)
    assert np.all(st.kc[il][:pos] == 0) and np.all(st.kc[il][pos + 1:] == 0)
    assert st.kv_len == pos + 1


def test_forward_token_with_silent_layers_is_embedding_lookup_and_lm_head():
    cfg = synth.CFG_TINY
    w = synth.make_model_weights(cfg)
    for L in w.layers:
        _zero(L.ffn_down)
        _zero(L.ssm_out if L.kind == synth.DELTANET else L.attn_output)
    m = oracle.Model(w)
    st = oracle.State(m)
    tok, hidden, logits = oracle.forward_token(m, st, 123, 0, want_logits=True)
    assert np.array_equal(hidden, w.token_embd[123])
    expect = oracle.gemv(w.lm_head, oracle.rmsnorm(w.token_embd[123], w.output_norm))
    assert np.array_equal(logits, expect)
    assert tok == int(np.argmax(expect))
    with pytest.raises(ValueError):
        oracle.forward_token(m, st, cfg.vocab, 0)
    with pytest.raises(ValueError):
        oracle.forward_token(m, st, 0, cfg.max_seq_len)
