"""Deterministic fixed-point softmax (DSM) used for every sampling decision.

What it computes.  The probability rule of "EAGLE-3: Engineering Implementation
of LLM Inference Acceleration", section X (``probs``: softmax(z / T), or the
one-hot argmax at T = 0) and the normalised residual of section X.5.  A float
softmax reduces in an order that differs between CPU and GPU, so a token drawn
from it is not reproducible bit for bit.  Reading taken here: every decision is
made on integer weights built by a fixed sequence of IEEE fp32
round-to-nearest operations, identical on both sides:

    m   = max_i z_i                             (exact compare)
    t_i = fp32(fp32(z_i - m) * invT)            invT = fp32(1 / T)
    w_i = EXP(t_i)                              in [0, 1]
    W_i = floor(w_i * 2**31)                    integer, W_i <= 2**31
    S   = sum_i W_i                             exact integer sum
    p_i = W_i / S                               the distribution that is used
    logq_i = fp32(t_i - LOG31(S))               LOG31(S) ~ ln(S * 2**-31)

Tokens with w_i < 2**-31 (logits more than about 21.5 nats below the row max)
get probability 0.

EXP: Cody-Waite reduction t = k ln2 + r with ln2 split into a 16-significant-bit
head and an fp32 tail, then the degree-7 Taylor polynomial of e^r (coefficients
fp32(1/j!)) in Horner form, then an exact scaling by 2**k.  Inputs below -64
give 0.  LOG31: S = 2**e * m with m the top 24 bits of S, m folded into
[sqrt(1/2), sqrt(2)), ln m = 2 s (1 + s^2/3 + ... + s^10/11) with
s = (m - 1)/(m + 1).  Every step is a separate RN fp32 op (no fused
multiply-add).

Pinned by: EXP against math.exp (relative error bound), LOG31 against
math.log, and p against the fp64 softmax (|p - softmax| <= V * 2**-31 + eps);
see tests/test_oracle_basics.py.
"""
import math

import numpy as np

f32 = np.float32

LN2_HI = f32(round(math.log(2.0) * 65536.0) / 65536.0)        # 16 significant bits
LN2_LO = f32(math.log(2.0) - float(LN2_HI))
LOG2E = f32(1.0 / math.log(2.0))
LN2 = f32(math.log(2.0))
SQRT2 = f32(math.sqrt(2.0))
EXP_C = [f32(1.0 / math.factorial(j)) for j in range(8)]       # 1/j!, j = 0..7
LOG_D = [f32(1.0 / j) for j in (1, 3, 5, 7, 9, 11)]           # 1/(2i+1)
EXP_MIN = f32(-64.0)
FIX_BITS = 31


def exp_f32(t):
    """EXP over an fp32 array of non-positive values (elementwise, RN fp32 ops)."""
    t = np.asarray(t, dtype=f32)
    with np.errstate(over="ignore", invalid="ignore", under="ignore"):
        k = np.rint(t * LOG2E).astype(f32)
        r = (t - k * LN2_HI).astype(f32)
        r = (r - k * LN2_LO).astype(f32)
        p = np.full_like(r, EXP_C[7])
        for j in range(6, -1, -1):
            p = (p * r).astype(f32)
            p = (p + EXP_C[j]).astype(f32)
        ki = np.where(t < EXP_MIN, 0, k).astype(np.int32)
        out = np.ldexp(p, ki).astype(f32)
    return np.where(t < EXP_MIN, f32(0.0), out).astype(f32)


def log31(S):
    """LOG31(S) ~ ln(S * 2**-31) in fp32, for a Python int S >= 1."""
    S = int(S)
    e = S.bit_length() - 1
    mant = S >> (e - 23) if e >= 23 else S << (23 - e)          # top 24 bits, truncated
    m = f32(f32(mant) * f32(2.0 ** -23))
    if m > SQRT2:
        m = f32(m * f32(0.5))
        e += 1
    s = f32(f32(m - f32(1.0)) / f32(m + f32(1.0)))
    s2 = f32(s * s)
    q = LOG_D[5]
    for j in range(4, -1, -1):
        q = f32(f32(q * s2) + LOG_D[j])
    lnm = f32(f32(f32(2.0) * s) * q)
    return f32(f32(f32(e - FIX_BITS) * LN2) + lnm)


def row_max(z):
    """Maximum of an fp32 row (finite values)."""
    return f32(np.max(np.asarray(z, dtype=f32)))


def scaled(z, inv_t):
    """t_i = fp32(fp32(z_i - m) * invT)."""
    z = np.asarray(z, dtype=f32)
    m = row_max(z)
    return ((z - m).astype(f32) * f32(inv_t)).astype(f32)


def inv_temperature(temperature):
    return f32(f32(1.0) / f32(temperature))


def weights(z, inv_t):
    """Integer weights W (int64 array, W_i <= 2**31) and their sum S (Python int)."""
    t = scaled(z, inv_t)
    w = exp_f32(t)
    W = np.floor(w.astype(np.float64) * float(2 ** FIX_BITS)).astype(np.int64)
    return W, int(W.sum())


def logq(z, inv_t=f32(1.0)):
    """Log-probabilities logq_i = fp32(t_i - LOG31(S)) for a whole row."""
    t = scaled(z, inv_t)
    _, S = weights(z, inv_t)
    return (t - log31(S)).astype(f32)


def probabilities(z, inv_t):
    """p_i = W_i / S as fp64 (for tests and reports; decisions use W, S)."""
    W, S = weights(z, inv_t)
    return W.astype(np.float64) / float(S)
