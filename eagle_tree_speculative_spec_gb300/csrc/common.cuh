// Shared device helpers: Philox4x32-10, the deterministic fixed-point softmax
// (EXP, LOG31), fp32 total order, status words, bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/eagle3.h"

#define E3_DEV __device__ __forceinline__

namespace e3 {

// ------------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11, section 3): ten rounds of two 32x32->64 multiplies with the key bumped by the Weyl
// constants between rounds.
// ------------------------------------------------------------------------------------------------
struct U4 {
    uint32_t x0, x1, x2, x3;
};

E3_DEV U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += W0;
            k1 += W1;
        }
        const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
        const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return U4{c0, c1, c2, c3};
}

// Counter layout of the acceptance stage: (slot + 256 * node, b, step lo, step hi), key = seed.
constexpr int SLOT_RESIDUAL = 64;
constexpr int SLOT_DRAW = 128;

E3_DEV U4 accept_draw(uint64_t seed, uint64_t step, int b, int node, int slot) {
    return philox4x32_10((uint32_t)slot + 256u * (uint32_t)node, (uint32_t)b, (uint32_t)step,
                         (uint32_t)(step >> 32), (uint32_t)seed, (uint32_t)(seed >> 32));
}

// ------------------------------------------------------------------------------------------------
// Deterministic fixed-point softmax.  Every step is an explicit IEEE fp32 round-to-nearest op
// (no contraction into FMA), so the result is bit-identical to a CPU that follows the same steps.
//   EXP(t), t <= 0: Cody-Waite reduction t = k ln2 + r with ln2 = LN2_HI + LN2_LO (LN2_HI has 16
//   significant bits so k * LN2_HI is exact), Taylor polynomial of e^r of degree 7 (coefficients
//   1/j! rounded to fp32) in Horner form, exact scaling by 2^k; t < -64 gives 0.
//   W = floor(EXP(t) * 2^31) as an integer (exact: a power-of-two scaling then truncation).
//   LOG31(S) ~ ln(S * 2^-31): S = 2^e * m with m the top 24 bits of S, folded into
//   [sqrt(1/2), sqrt(2)); ln m = 2 s (1 + s^2/3 + ... + s^10/11), s = (m - 1) / (m + 1).
// ------------------------------------------------------------------------------------------------
constexpr int FIX_BITS = 31;
constexpr float LN2_HI = 0x1.62e4p-1f;        // ln 2 rounded to 16 significant bits
constexpr float LN2_LO = 0x1.7f7d1cp-20f;     // fp32(ln 2 - LN2_HI)
constexpr float LOG2E = 0x1.715476p+0f;       // fp32(1 / ln 2)
constexpr float LN2_F = 0x1.62e43p-1f;        // fp32(ln 2)
constexpr float SQRT2_F = 0x1.6a09e6p+0f;     // fp32(sqrt 2)

E3_DEV float dsm_exp(float t) {
    if (!(t >= -64.0f)) return 0.0f;   // also catches NaN and -inf
    const float k = rintf(__fmul_rn(t, LOG2E));
    float r = __fsub_rn(t, __fmul_rn(k, LN2_HI));
    r = __fsub_rn(r, __fmul_rn(k, LN2_LO));
    float p = 0x1.a01a02p-13f;                 // 1/7!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.6c16c2p-10f);   // 1/6!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.111112p-7f);    // 1/5!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-5f);     // 1/4!
    p = __fadd_rn(__fmul_rn(p, r), 0x1.555556p-3f);      // 1/3!
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const int ki = (int)k;                                    // in [-93, 0]
    return __fmul_rn(p, __int_as_float((ki + 127) << 23));    // exact: normal power of two
}

// t_i = fp32(fp32(z_i - m) * invT)
E3_DEV float dsm_scaled(float z, float m, float inv_t) { return __fmul_rn(__fsub_rn(z, m), inv_t); }

E3_DEV uint32_t dsm_weight(float t) {
    // EXP(t) * 2^31 <= 2^31 is exact in fp32; truncation to an integer is the floor (t <= 0 -> >= 0)
    return (uint32_t)__fmul_rn(dsm_exp(t), 2147483648.0f);
}

// dsm_weight(dsm_scaled(z, m, inv_t)) for two values at once.  The same RN operations run lane by
// lane on paired fp32 multiplies and adds (no fusion; a - b is computed as a + (-b), which IEEE
// rounding makes identical), so each weight is bit-identical to the scalar path.
E3_DEV uint2 dsm_weight_pair(float z0, float z1, float m, float inv_t) {
    auto dup = [](float x) { return make_float2(x, x); };
    auto neg = [](float2 x) { return make_float2(-x.x, -x.y); };
    const float2 t = __fmul2_rn(__fadd2_rn(make_float2(z0, z1), dup(-m)), dup(inv_t));
    // below -64 (or NaN) the weight is 0; clamp so that the exponent arithmetic stays in range
    const float2 tc = make_float2(fmaxf(t.x, -64.0f), fmaxf(t.y, -64.0f));
    const float2 kl = __fmul2_rn(tc, dup(LOG2E));
    const float2 k = make_float2(rintf(kl.x), rintf(kl.y));
    float2 r = __fadd2_rn(tc, neg(__fmul2_rn(k, dup(LN2_HI))));
    r = __fadd2_rn(r, neg(__fmul2_rn(k, dup(LN2_LO))));
    float2 q = dup(0x1.a01a02p-13f);                       // 1/7!
    q = __fadd2_rn(__fmul2_rn(q, r), dup(0x1.6c16c2p-10f));   // 1/6!
    q = __fadd2_rn(__fmul2_rn(q, r), dup(0x1.111112p-7f));    // 1/5!
    q = __fadd2_rn(__fmul2_rn(q, r), dup(0x1.555556p-5f));    // 1/4!
    q = __fadd2_rn(__fmul2_rn(q, r), dup(0x1.555556p-3f));    // 1/3!
    q = __fadd2_rn(__fmul2_rn(q, r), dup(0.5f));
    q = __fadd2_rn(__fmul2_rn(q, r), dup(1.0f));
    q = __fadd2_rn(__fmul2_rn(q, r), dup(1.0f));
    const float2 e = __fmul2_rn(q, make_float2(__int_as_float(((int)k.x + 127) << 23),
                                               __int_as_float(((int)k.y + 127) << 23)));
    const float2 w = __fmul2_rn(e, dup(2147483648.0f));
    return make_uint2(t.x >= -64.0f ? (uint32_t)w.x : 0u, t.y >= -64.0f ? (uint32_t)w.y : 0u);
}

E3_DEV int bitlen64(uint64_t v) { return v ? 64 - __clzll((long long)v) : 0; }

E3_DEV float dsm_log31(uint64_t S) {
    int e = bitlen64(S) - 1;
    const uint64_t mant = e >= 23 ? (S >> (e - 23)) : (S << (23 - e));   // in [2^23, 2^24)
    float m = __fmul_rn((float)(uint32_t)mant, 0x1p-23f);                 // exact
    if (m > SQRT2_F) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
    const float s2 = __fmul_rn(s, s);
    float q = 0x1.745d18p-4f;                   // 1/11
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.c71c72p-4f);      // 1/9
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.24924ap-3f);      // 1/7
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.99999ap-3f);      // 1/5
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.555556p-2f);      // 1/3
    q = __fadd_rn(__fmul_rn(q, s2), 1.0f);
    const float lnm = __fmul_rn(__fmul_rn(2.0f, s), q);
    return __fadd_rn(__fmul_rn((float)(e - FIX_BITS), LN2_F), lnm);
}

// EXP_NOISE(w): an Exp(1) draw from a 32-bit word.  u = (2 (w >> 9) + 1) * 2^-24 (odd numerator
// S < 2^24, exact in fp32); S = 2^e * m folded into [sqrt(1/2), sqrt(2)) as in dsm_log31, and
// E = (24 - e) ln 2 - ln m = -ln u with the same atanh series and RN steps (no cancellation near
// u = 1, and E > 0 for every w).
E3_DEV float dsm_exp_noise(uint32_t w) {
    const uint32_t S = 2u * (w >> 9) + 1u;
    int e = 31 - __clz(S);                                                 // bit length - 1
    float m = __fmul_rn((float)S, __int_as_float((127 - e) << 23));        // exact: S < 2^24
    if (m > SQRT2_F) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
    const float s2 = __fmul_rn(s, s);
    float q = 0x1.745d18p-4f;                   // 1/11
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.c71c72p-4f);      // 1/9
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.24924ap-3f);      // 1/7
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.99999ap-3f);      // 1/5
    q = __fadd_rn(__fmul_rn(q, s2), 0x1.555556p-2f);      // 1/3
    q = __fadd_rn(__fmul_rn(q, s2), 1.0f);
    const float lnm = __fmul_rn(__fmul_rn(2.0f, s), q);
    return __fsub_rn(__fmul_rn((float)(24 - e), LN2_F), lnm);
}

// ------------------------------------------------------------------------------------------------
// Total order on fp32 bit patterns: a > b as floats <=> key(a) > key(b) (and +0 > -0, NaN on top).
// Packed with the index so that the maximum of the packed value is the maximum key with the
// lowest index.
// ------------------------------------------------------------------------------------------------
E3_DEV uint32_t order_key(float z) {
    const int32_t i = __float_as_int(z);
    const int32_t k = i < 0 ? (i ^ 0x7FFFFFFF) : i;
    return (uint32_t)k ^ 0x80000000u;   // signed order -> unsigned order
}
E3_DEV float key_to_float(uint32_t u) {
    const int32_t k = (int32_t)(u ^ 0x80000000u);
    return __int_as_float(k < 0 ? (k ^ 0x7FFFFFFF) : k);
}
E3_DEV uint64_t pack_argmax(float z, uint32_t idx) {
    return ((uint64_t)order_key(z) << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}
E3_DEV uint32_t unpack_idx(uint64_t p) { return 0xFFFFFFFFu - (uint32_t)p; }

// ------------------------------------------------------------------------------------------------
// Status words and bounded waits.
// ------------------------------------------------------------------------------------------------
E3_DEV void flag(int32_t *dev_status, int bits) {
    if (dev_status) atomicOr(dev_status, bits);
}

// ~2 s at 2 GHz: a wait that outlives this has lost its producer
constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;

E3_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ------------------------------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with launch_pdl may be dispatched while the
// previous kernel of its stream retires its last blocks; it runs pdl_wait() before its first
// global memory access, which returns once that kernel has completed and its writes are visible
// (for an ordinary launch it returns at once).  pdl_trigger() lets the next kernel be dispatched
// before this one ends: its blocks take SMs as this kernel's blocks retire and run their prologue
// there (barrier setup, TMEM allocation) up to their own pdl_wait().  The next kernel is dispatched
// only once every block of this one has triggered or exited, so its blocks never hold resources
// that a block of this kernel still waits for; its pdl_wait() still waits for this whole kernel.
// ------------------------------------------------------------------------------------------------
E3_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
E3_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Host-side value computed once per device (for the device current at the call) and kept:
// kernel attributes and device attribute queries.  Safe for concurrent callers.
template <typename T>
struct PerDevice {
    static constexpr int MAX_DEVICES = 128;
    std::mutex mu;
    bool done[MAX_DEVICES] = {};
    T val[MAX_DEVICES] = {};
    template <typename F>
    T get(F f) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return f();
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            val[dev] = f();
            done[dev] = true;
        }
        return val[dev];
    }
};

// SMs of the current device, 0 when it cannot be queried (no device)
inline int device_sm_count() {
    static PerDevice<int> cache;
    return cache.get([] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            n = 0;
        return n > 0 ? n : 0;
    });
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace e3
