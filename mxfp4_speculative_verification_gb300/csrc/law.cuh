// The sampling law of one logit row, as the kernels of law.cu compute it and
// as spec_accept evaluates it from logits ("Module 11. Speculative Decoding
// and Quantization", §4: acceptance uses the laws tokens are actually sampled
// from, after temperature, top-k and top-p, on the target and the draft
// alike).  Shared by law.cu and accept.cu so that the probabilities written
// out and the ones the acceptance kernel forms on the fly are the same bits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxs {

// Per-row statistics of a transformed law: token t is kept iff
// law_key(logit_t) >= cut, and then p_t = exp((logit_t - m) / T) * inv_s.
struct LawStats {
    float m;        // largest finite logit of the row
    uint32_t cut;   // smallest kept key (top-k and top-p thresholds together)
    float inv_s;    // 2^46 / (sum over kept tokens of floor(exp(...) * 2^46))
    int32_t ok;     // 0: the row has no law (a NaN or +inf logit, or nothing finite)
};

// Monotone image of an fp32 value in uint32 (larger value, larger key).
__device__ __forceinline__ uint32_t law_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Unnormalised mass of a logit: exp((l - m) / T), in [0, 1] for l <= m, by
// the fast exponential intrinsic (its error grows with the argument: ~1e-7
// relative at the top of the law, ~1e-6 ten nats below it).
__device__ __forceinline__ float law_exp(float l, float m, float inv_t) { return __expf((l - m) * inv_t); }

// The transformed law's probability of a token with logit l.
__device__ __forceinline__ float law_value(float l, const LawStats& s, float inv_t) {
    if (!s.ok || law_key(l) < s.cut) return 0.f;
    return law_exp(l, s.m, inv_t) * s.inv_s;
}

// Fixed-point mass of one token, floor(e * 2^46) for e in [0, 1]: sums of
// these are exact in any order, so the top-p cut does not depend on which
// thread added what.  Formed as two 23-bit digits by exact fp32 operations
// (cheaper than 64-bit integer shifts): y = e 2^23 (exact), the add y + 2^23
// rounded toward zero holds 2^23 + floor(y), whose bit pattern is
// kMassBias + floor(y); the fraction y - floor(y) is exact, and the same add
// on it times 2^23 gives the low digit.  floor(e 2^46) = hi 2^23 + lo, equal
// to the integer definition for every float in [0, 1].
constexpr uint32_t kMassBias = 0x4B000000u;  // the bit pattern of 2^23

// The two digits, each still carrying kMassBias (callers subtract it, often
// inside an accumulation).
__device__ __forceinline__ void law_mass_digits(float e, uint32_t& hb, uint32_t& lb) {
    const float two23 = 8388608.f;
    const float y = __fmul_rn(e, two23);
    const float t = __fadd_rz(y, two23);
    const float z = __fmul_rn(__fsub_rn(y, __fsub_rn(t, two23)), two23);
    hb = __float_as_uint(t);
    lb = __float_as_uint(__fadd_rz(z, two23));
}

__device__ __forceinline__ unsigned long long law_mass(float e) {
    uint32_t hb, lb;
    law_mass_digits(e, hb, lb);
    return (static_cast<unsigned long long>(hb - kMassBias) << 23) + (lb - kMassBias);
}

}  // namespace mxs
