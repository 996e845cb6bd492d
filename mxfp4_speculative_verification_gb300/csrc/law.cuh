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
// thread added what.  Taken from the bits (a normal e is M * 2^(E - 150), M
// its 24-bit significand, E its biased exponent, so e * 2^46 = M * 2^(E - 104);
// zero and subnormal e give 0), which measured faster here than the 64-bit
// float-to-integer conversion.
__device__ __forceinline__ unsigned long long law_mass(float e) {
    const uint32_t b = __float_as_uint(e);
    const int E = int(b >> 23);
    const unsigned long long M = (b & 0x7FFFFFu) | 0x800000u;
    const int sh = E - 104;
    if (E == 0 || sh <= -24) return 0ull;
    return sh >= 0 ? M << sh : M >> -sh;
}

}  // namespace mxs
