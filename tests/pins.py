"""Pin checks for the oracle's arithmetic, shared by the pin tests and the planted-mistake tests.

Each ``pin_*`` function raises AssertionError when the oracle (looked up at
call time, so a test may patch it) disagrees with something the pages or the
mathematics fix independently of the oracle's own code.
"""

import math
from fractions import Fraction

import numpy as np

from oracle import numerics, steps

HP = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}


def rand_bf16(rng, n, sigma):
    return numerics.bf16_rne((rng.standard_normal(n) * sigma).astype(np.float32))


def f32(x):
    return float(np.float32(x))


# ---------------------------------------------------------------- bf16 by enumeration

_POS_BF16 = None


def _positive_bf16_values():
    """All finite non-negative bf16 values in increasing order (as Fractions), with their bits."""
    global _POS_BF16
    if _POS_BF16 is None:
        bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
        vals = numerics.f32_from_bf16(bits).astype(np.float64)
        _POS_BF16 = (vals, bits)
    return _POS_BF16


def bf16_nearest_even_of_fraction(x: Fraction) -> int:
    """bf16 bits of the exact rational x rounded to nearest, ties to even, found by search."""
    vals, bits = _positive_bf16_values()
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    j = int(np.searchsorted(vals, float(a)))
    best = None
    for cand in range(max(0, j - 2), min(len(vals), j + 3)):
        d = abs(Fraction(vals[cand]) - a)
        if best is None or d < best[0] or (d == best[0] and int(bits[cand]) % 2 == 0):
            best = (d, cand)
    return int(bits[best[1]]) | sign


# ---------------------------------------------------------------- accumulation

def pin_accumulation_four_equal_microbatches():
    """4 equal micro-batch gradients, each scaled by 1/4 before accumulation, give the full-batch mean.

    Full-batch mean of four copies of g is g itself.  Checked on every bf16
    pattern whose quarter is a normal number.
    """
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = numerics.f32_from_bf16(bits)
    finite = np.isfinite(g)
    bits, g = bits[finite], g[finite]
    normal_quarter = np.abs(g.astype(np.float64)) >= 2.0 ** -124
    acc = None
    for j in range(4):
        acc = steps.accumulate(acc, bits, 0.25, first=(j == 0))
    assert np.array_equal(acc[normal_quarter], bits[normal_quarter])
    # +0 and -0 both accumulate to +0 (the buffer starts from +0)
    zero_sel = (bits == 0) | (bits == 0x8000)
    assert np.all(acc[zero_sel] == 0)


def pin_accumulation_linear_model():
    """Gradient accumulation of a least-squares model equals its full-batch gradient.

    The loss is the sample mean over 16 samples; 4 equal micro-batches of 4
    samples each give micro-batch mean gradients; scaling each by 1/4 and
    summing must give the full-batch gradient, up to the bf16 roundings
    (inputs and four accumulation steps: at most 3 ulps of the largest partial sum).
    """
    rng = np.random.default_rng(3)
    X = rng.standard_normal((16, 12))
    y = rng.standard_normal(16)
    w = rng.standard_normal(12) * 0.1
    full = X.T @ (X @ w - y) / 16.0
    acc = None
    partial_max = np.zeros(12)
    running = np.zeros(12)
    for j in range(4):
        Xj, yj = X[4 * j:4 * j + 4], y[4 * j:4 * j + 4]
        gj = Xj.T @ (Xj @ w - yj) / 4.0
        gj_bits = numerics.bf16_rne(gj.astype(np.float32))
        acc = steps.accumulate(acc, gj_bits, 0.25, first=(j == 0))
        running = running + gj / 4.0
        partial_max = np.maximum(partial_max, np.abs(running))
    got = numerics.f32_from_bf16(acc).astype(np.float64)
    tol = 3.0 * partial_max * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(got - full) <= tol), (got, full)


# ---------------------------------------------------------------- mean over ranks

def pin_mean_against_exact_rationals(seed=5):
    """Reduce-with-average on tiny buffers vs the exact rational mean.

    Where the fp32 sum is exact (checked with Fractions) the result must be
    the exact mean rounded once to bf16; otherwise it may differ from that by
    at most one bf16 ulp.
    """
    rng = np.random.default_rng(seed)
    for n_d in (1, 2, 3, 4, 5, 8):
        for _ in range(40):
            grads = [rand_bf16(rng, 6, 10.0 ** rng.uniform(-6, 1)) for _ in range(n_d)]
            got = steps.reduce_mean(grads)
            for i in range(6):
                vals = [Fraction(float(numerics.f32_from_bf16(g[i:i + 1])[0])) for g in grads]
                exact_sum = sum(vals, Fraction(0))
                want = bf16_nearest_even_of_fraction(exact_sum / n_d)
                fp32_sum = np.float32(0)
                for v in vals:
                    fp32_sum = np.float32(fp32_sum + np.float32(float(v)))
                if Fraction(float(fp32_sum)) == exact_sum and n_d in (1, 2, 4, 8):
                    assert int(got[i]) == want, (n_d, i, vals)
                else:
                    gv = float(numerics.f32_from_bf16(got[i:i + 1])[0])
                    wv = float(numerics.f32_from_bf16(np.array([want], dtype=np.uint16))[0])
                    ulp = float(numerics.bf16_ulp(np.array([want], dtype=np.uint16))[0])
                    assert abs(gv - wv) <= ulp, (n_d, i, gv, wv)


def pin_mean_of_equal_grads():
    rng = np.random.default_rng(9)
    g = rand_bf16(rng, 4096, 1e-3)
    for n_d in (1, 2, 4, 8, 16, 32):
        assert np.array_equal(steps.reduce_mean([g] * n_d), g)


# ---------------------------------------------------------------- AdamW

def pin_adamw_first_step_closed_form():
    """t = 1 from m = v = 0: bias correction gives m_hat = g and v_hat = g^2, so
    p1 = p0*(1 - lr*wd) - lr * g / (|g| + eps), evaluated in float64 and compared
    within a few fp32 rounding errors."""
    rng = np.random.default_rng(1)
    n = 20000
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g_bits = rand_bf16(rng, n, 1e-3)
    g = numerics.f32_from_bf16(g_bits).astype(np.float64)
    z = np.zeros(n, np.float32)
    p1, m1, v1, bits = steps.adamw(p0, z, z, g_bits, HP, 1)
    lr, wd, eps = f32(HP["lr"]), f32(HP["weight_decay"]), f32(HP["eps"])
    b1, b2 = f32(HP["beta1"]), f32(HP["beta2"])
    want = p0.astype(np.float64) * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    tol = 8 * 2.0 ** -24 * (np.abs(p0.astype(np.float64)) + lr)
    assert np.all(np.abs(p1.astype(np.float64) - want) <= tol)
    assert np.allclose(m1, (1 - b1) * g, rtol=3e-7, atol=0)
    assert np.allclose(v1, (1 - b2) * g * g, rtol=5e-7, atol=0)
    assert np.array_equal(bits, numerics.bf16_rne(p1))


def pin_adamw_zero_stays_zero():
    """Padding elements: zero gradient, zero master, zero moments stay exactly zero."""
    z = np.zeros(64, np.float32)
    g = np.zeros(64, np.uint16)
    p, m, v = z, z, z
    for t in range(1, 30):
        p, m, v, bits = steps.adamw(p, m, v, g, HP, t)
        assert not p.any() and not m.any() and not v.any() and not bits.any()


def pin_adamw_weight_decay_only():
    """With g = 0 the moments stay 0 and p_t = p_0 * (1 - lr*wd)^t (decoupled decay)."""
    rng = np.random.default_rng(2)
    p0 = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    z = np.zeros(1000, np.float32)
    g = np.zeros(1000, np.uint16)
    p, m, v = p0, z, z
    T = 10
    for t in range(1, T + 1):
        p, m, v, _ = steps.adamw(p, m, v, g, HP, t)
    decay = 1 - f32(HP["lr"]) * f32(HP["weight_decay"])
    want = p0.astype(np.float64) * decay ** T
    assert np.all(np.abs(p - want) <= (T + 1) * 2.0 ** -24 * np.abs(want))
    assert not m.any() and not v.any()


def pin_adamw_float64_shadow(steps_n=10):
    """Each fp32 step against the same step in float64 from the same fp32 inputs.

    Every quantity of one step is a short chain of rounded operations, so the
    fp32 result is within a few ulps of the float64 one (relative to the
    magnitudes involved)."""
    rng = np.random.default_rng(4)
    n = 20000
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    lr, wd, eps = f32(HP["lr"]), f32(HP["weight_decay"]), f32(HP["eps"])
    b1, b2 = f32(HP["beta1"]), f32(HP["beta2"])
    u = 2.0 ** -24
    for t in range(1, steps_n + 1):
        g_bits = rand_bf16(rng, n, 1e-3)
        g = numerics.f32_from_bf16(g_bits).astype(np.float64)
        P, M, V = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
        M1 = b1 * M + (1 - b1) * g
        V1 = b2 * V + (1 - b2) * g * g
        den = np.sqrt(V1) / math.sqrt(1 - b2 ** t) + eps
        P1 = P * (1 - lr * wd) - (lr / (1 - b1 ** t)) * M1 / den
        p, m, v, _ = steps.adamw(p, m, v, g_bits, HP, t)
        mag_m = b1 * np.abs(M) + (1 - b1) * np.abs(g)
        assert np.all(np.abs(m - M1) <= 4 * u * mag_m)
        assert np.all(np.abs(v - V1) <= 4 * u * V1 + 1e-45)
        # m carries an error of up to 4u * mag_m into the ratio; the denominator about 7u
        ratio_mag = (lr / (1 - b1 ** t)) * (mag_m + np.abs(M1)) / den
        assert np.all(np.abs(p - P1) <= 4 * u * np.abs(P) + 12 * u * ratio_mag)


def pin_adamw_against_torch(steps_n=10):
    """Agreement with torch.optim.AdamW (CPU, fp32, single-tensor), step by step.

    Before each step torch is given the oracle's current state, so the
    comparison measures one step.  torch arranges some operations differently
    (a lerp for m, addcmul for v, addcdiv for the update), so agreement is to
    a few fp32 roundings of each quantity's operands."""
    import torch

    rng = np.random.default_rng(6)
    n = 50000
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    param = torch.nn.Parameter(torch.from_numpy(p.copy()))
    # the same fp32 hyper-parameter values the oracle uses, handed to torch as Python floats
    opt = torch.optim.AdamW([param], lr=f32(HP["lr"]), betas=(f32(HP["beta1"]), f32(HP["beta2"])),
                            eps=f32(HP["eps"]), weight_decay=f32(HP["weight_decay"]),
                            foreach=False, fused=False)
    u = 2.0 ** -24
    for t in range(1, steps_n + 1):
        g_bits = rand_bf16(rng, n, 1e-3)
        g = numerics.f32_from_bf16(g_bits)
        with torch.no_grad():
            param.copy_(torch.from_numpy(p))
        if t > 1:
            st = opt.state[param]
            st["exp_avg"].copy_(torch.from_numpy(m))
            st["exp_avg_sq"].copy_(torch.from_numpy(v))
        param.grad = torch.from_numpy(g.copy())
        opt.step()
        prev = p
        p, m1, v1, _ = steps.adamw(p, m, v, g_bits, HP, t)
        st = opt.state[param]
        assert int(st["step"]) == t
        tp = param.detach().numpy()
        tm = st["exp_avg"].numpy()
        tv = st["exp_avg_sq"].numpy()
        # moments: a few roundings of their inputs.  master: a few ulps of the operands of the
        # last subtraction, plus what the m difference and a few roundings do to the update
        err_m = 4 * u * (np.abs(m) + np.abs(g))
        assert np.all(np.abs(m1 - tm) <= err_m)
        den = np.sqrt(v1.astype(np.float64)) / math.sqrt(1 - f32(HP["beta2"]) ** t) + f32(HP["eps"])
        step_size = f32(HP["lr"]) / (1 - f32(HP["beta1"]) ** t)
        err_upd = step_size * (err_m + 8 * u * np.abs(m1)) / den
        assert np.all(np.abs(p - tp) <= 4 * u * (np.abs(prev) + np.abs(tp)) + err_upd)
        assert np.all(np.abs(v1 - tv) <= 4 * u * np.abs(tv))
        m, v = m1, v1


def pin_sharded_update_equals_unsharded():
    """AdamW is element-wise: updating the N_d shards separately and concatenating
    equals updating the whole buffer at once, bit for bit."""
    rng = np.random.default_rng(8)
    n_d, S = 4, 3001
    n = n_d * S
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-7).astype(np.float32)
    g = rand_bf16(rng, n, 1e-3)
    whole = steps.adamw(p, m, v, g, HP, 3)
    parts = [steps.adamw(p[r * S:(r + 1) * S], m[r * S:(r + 1) * S], v[r * S:(r + 1) * S],
                         g[r * S:(r + 1) * S], HP, 3) for r in range(n_d)]
    for j in range(4):
        assert np.array_equal(np.concatenate([pt[j] for pt in parts]), whole[j])


ALL_ADAMW_PINS = [
    pin_adamw_first_step_closed_form,
    pin_adamw_zero_stays_zero,
    pin_adamw_weight_decay_only,
    pin_adamw_float64_shadow,
    pin_adamw_against_torch,
]
