// Per-lane quantization core shared by the standalone quantizer kernels and
// the quantizing prologue of the fused GEMM, so that both produce identical
// codes and scale bytes.
//
// ResServe App. B.2 Eq. 8-10 and Algorithm 1 (eight inputs per lane): the
// lanes that share one scale block (2 for NVFP4's 16-element blocks, 4 for
// MXFP4's 32-element blocks) combine their maxima with shuffles, every lane
// derives the block scale and the fp32 multiplier, converts its eight values
// to E2M1, and decodes them again to form the reconstruction x^ (and from it
// the residue) in registers.
#pragma once

#include "rs_device.cuh"

namespace rs {

// NVFP4 block scale from the block amax (Eq. 8-9, Alg. 1 line 3):
// byte = E4M3(fl(fl(amax/6)/alpha)), s~ = fl(alpha * dec(byte)), mul = fl(1/s~).
__device__ __forceinline__ uint32_t nv_block_scale(float amax, float alpha, float& st, float& mul) {
    const float s = __fdiv_rn(amax, kE2M1Max);
    const float t = alpha > 0.0f ? __fdiv_rn(s, alpha) : 0.0f;
    const uint32_t sf = e4m3_encode_satfinite(t);
    st = __fmul_rn(alpha, e4m3_decode(sf));
    mul = st == 0.0f ? 0.0f : __fdiv_rn(1.0f, st);
    return sf;
}

// NVFP4 tensor scales the quantizers support: 0, or finite and at least
// 2^-117, so that every non-zero block scale s~ >= alpha * 2^-9 is a normal
// float and fl(1/s~) is finite.  (Below that, x * fl(1/s~) can be infinite
// or NaN and the E2M1 rounding of Eq. 10 is undefined.)
__device__ __forceinline__ bool nv_alpha_supported(float alpha) {
    return alpha == 0.0f || (alpha >= 0x1p-117f && alpha <= 3.40282347e38f);
}

// Per-tensor constants of the fast NVFP4 scale path: c = fl(1/fl(6 alpha)),
// usable when alpha > 0 and c is a normal float.
struct NvScaleConst {
    float alpha, c;
    bool fast;
};
__device__ __forceinline__ NvScaleConst nv_scale_const(float alpha) {
    NvScaleConst k;
    k.alpha = alpha;
    k.c = alpha > 0.0f ? __frcp_rn(__fmul_rn(6.0f, alpha)) : 0.0f;
    k.fast = alpha > 0.0f && k.c >= 0x1p-126f && k.c < 0x1p126f;
    return k;
}

// Same result as nv_block_scale, with the divisions only where they decide.
// The estimate t~ = fl(amax * c) is within a relative 2^-21 of
// t = fl(fl(amax/6)/alpha) (five roundings of at most 2^-24 each, which
// needs fl(6 alpha), c and amax/6 to be normal floats: amax >= 2^-123);
// E4M3 rounding is monotone, so when both ends of the band t~(1 -+ 2^-20)
// round to the same byte, t rounds to it too.  t~ >= 448 means t >= 432,
// which rounds to the largest byte.  Blocks whose t lies within about 2^-20
// of a rounding boundary (a fraction of about 2^-16 of blocks) take the exact
// path.  st = fl(alpha * dec(byte)) and mul = fl(1/st) as in nv_block_scale
// (__frcp_rn is the correctly rounded reciprocal).
__device__ __forceinline__ uint32_t nv_block_scale_fast(float amax, const NvScaleConst& k, float& st, float& mul) {
    if (!k.fast || !(amax >= 0x1p-123f)) return nv_block_scale(amax, k.alpha, st, mul);
    const float t = __fmul_rn(amax, k.c);
    uint32_t sf;
    if (!(t < 448.0f)) {
        sf = 0x7Eu;
    } else {
        const uint32_t pr = e4m3x2_encode_hw(__fmul_rn(t, 1.0f - 0x1p-20f), __fmul_rn(t, 1.0f + 0x1p-20f));
        sf = pr & 0xFFu;
        if (sf != (pr >> 8)) return nv_block_scale(amax, k.alpha, st, mul);
    }
    st = __fmul_rn(k.alpha, e4m3_decode_hw(sf));
    mul = st == 0.0f ? 0.0f : __frcp_rn(st);
    return sf;
}

// The byte of nv_block_scale_fast alone (the caller looks up s~ and fl(1/s~)
// for it, e.g. in a table built with nv_scale_table_entry).
__device__ __forceinline__ uint32_t nv_block_byte(float amax, const NvScaleConst& k) {
    float st, mul;
    if (!k.fast || !(amax >= 0x1p-123f)) return nv_block_scale(amax, k.alpha, st, mul);
    const float t = __fmul_rn(amax, k.c);
    if (!(t < 448.0f)) return 0x7Eu;
    const uint32_t pr = e4m3x2_encode_hw(__fmul_rn(t, 1.0f - 0x1p-20f), __fmul_rn(t, 1.0f + 0x1p-20f));
    const uint32_t sf = pr & 0xFFu;
    if (sf != (pr >> 8)) return nv_block_scale(amax, k.alpha, st, mul);
    return sf;
}

// s~ = fl(alpha * dec(byte)) and mul = fl(1/s~) (0 when s~ == 0) for one of
// the 127 finite non-negative E4M3 bytes: the values nv_block_scale gives.
__device__ __forceinline__ void nv_scale_table_entry(uint32_t byte, float alpha, float& st, float& mul) {
    st = byte < 127u ? __fmul_rn(alpha, e4m3_decode_hw(byte)) : 0.0f;
    mul = st == 0.0f ? 0.0f : __frcp_rn(st);
}

// max(|x|) over the sixteen bf16 values of eight words, ignoring NaN like
// fmaxf and starting from +0 (bf16 -> fp32 is exact, so the order is the
// fp32 one); two values per max.bf16x2.
__device__ __forceinline__ float amax16_bf16(const uint32_t (&w)[8]) {
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i] & 0x7FFF7FFFu));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// MXFP4 block scale: byte = max(E - 2, 0) where E is the biased fp32
// exponent of amax, i.e. e = floor(log2 amax) - 2 clamped at -127 (amax == 0
// and fp32-subnormal amax give byte 0).  st = 2^e, mul = 2^-e, both exact.
__device__ __forceinline__ uint32_t mx_block_scale(float amax, float& st, float& mul) {
    const int E = (int)(__float_as_uint(amax) >> 23);
    const uint32_t byte = E >= 2 ? (uint32_t)(E - 2) : 0u;
    st = byte >= 1u ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);  // 2^(byte-127)
    mul = __uint_as_float((254u - byte) << 23);                                      // 2^(127-byte)
    return byte;
}

// Shuffle-max over the lanes that share one scale block (full warp active).
template <int FMT>
__device__ __forceinline__ float block_amax(float a) {
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    if (FMT == 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    return a;
}

// Quantize this lane's eight values; returns the packed codes (element e in
// bits 4e..4e+3, i.e. element 2j in the low nibble of byte j), the block's
// scale byte in `sf`, and the reconstruction fl(s~ * dec(q)) in `xh`.
template <int FMT, bool kRecon = true>
__device__ __forceinline__ uint32_t quant_lane(const float (&xf)[8], const NvScaleConst& k, uint32_t& sf,
                                               float (&xh)[8]) {
    float am = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) am = fmaxf(am, fabsf(xf[e]));
    am = block_amax<FMT>(am);
    float st, mul;
    sf = FMT == 0 ? nv_block_scale_fast(am, k, st, mul) : mx_block_scale(am, st, mul);
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; e += 2) fmul2_rn(xf[e], xf[e + 1], mul, mul, v[e], v[e + 1]);
    const uint32_t codes = e2m1_encode8(v);
    if constexpr (kRecon) {  // the reconstruction is only needed to form a residue
        float d[8];
        e2m1_decode8(codes, d);
#pragma unroll
        for (int e = 0; e < 8; ++e) xh[e] = __fmul_rn(st, d[e]);
    }
    return codes;
}

// Residue of this lane's eight values, r = fl(x - x^) (Alg. 1 line 6).  The
// reconstruction and the residue use the scalar round-to-nearest intrinsics,
// which are never merged into a multiply-add: a fused x - s~ dec(q) rounds
// once and can move a residue code across an E2M1 rounding boundary.
__device__ __forceinline__ void residue8(const float (&xf)[8], const float (&xh)[8], float (&r)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = __fsub_rn(xf[e], xh[e]);
}

// Gather the four scale bytes of one atom row (4 consecutive blocks) into the
// first lane of its group: NVFP4 groups are 8 lanes (2 per block), MXFP4
// groups 16 lanes (4 per block).  Returns the word on every lane; only the
// group leader's copy is meaningful.
template <int FMT>
__device__ __forceinline__ uint32_t gather_sf_word(uint32_t sfbyte, int lane) {
    constexpr int kLanesPerBlock = FMT == 0 ? 2 : 4;
    constexpr int kLanesPerAtom = 4 * kLanesPerBlock;
    const int base = lane & ~(kLanesPerAtom - 1);
    const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, sfbyte, base);
    const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, sfbyte, base + kLanesPerBlock);
    const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, sfbyte, base + 2 * kLanesPerBlock);
    const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, sfbyte, base + 3 * kLanesPerBlock);
    return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

template <int FMT>
__host__ __device__ constexpr int lanes_per_atom() { return FMT == 0 ? 8 : 16; }

// One whole scale block per thread (16 elements NVFP4, 32 MXFP4): the block
// amax, scale and multiplier are computed once, and the E element codes come
// back packed 8 per 32-bit word (element e of the block in bits 4(e%8).. of
// word e/8).  Same arithmetic per element as quant_lane; the amax is a max,
// so its evaluation order does not change it.
template <int FMT, int E, bool kRecon = true>
__device__ __forceinline__ void quant_block(const float (&xf)[E], const NvScaleConst& k, uint32_t& sf,
                                            uint32_t (&codes)[E / 8], float (&xh)[E]) {
    float am0 = 0.0f, am1 = 0.0f;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        am0 = fmaxf(am0, fabsf(xf[e]));
        am1 = fmaxf(am1, fabsf(xf[e + 1]));
    }
    const float am = fmaxf(am0, am1);
    float st, mul;
    sf = FMT == 0 ? nv_block_scale_fast(am, k, st, mul) : mx_block_scale(am, st, mul);
#pragma unroll
    for (int w = 0; w < E / 8; ++w) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2) fmul2_rn(xf[8 * w + e], xf[8 * w + e + 1], mul, mul, v[e], v[e + 1]);
        codes[w] = e2m1_encode8(v);
        if constexpr (kRecon) {  // the reconstruction is only needed to form a residue
            float d[8];
            e2m1_decode8(codes[w], d);
#pragma unroll
            for (int e = 0; e < 8; ++e) xh[8 * w + e] = __fmul_rn(st, d[e]);
        }
    }
}

// max(|x|) over the bf16 values of W 32-bit words (two per word), as
// amax16_bf16 does for eight words.
template <int W>
__device__ __forceinline__ float amax_bf16_words(const uint32_t* w) {
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < W; ++i) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[i] & 0x7FFF7FFFu));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// One whole block (E = 16 NVFP4 / 32 MXFP4 elements) straight from its raw
// bf16 words: base codes and scale byte, and with kResidue the residue
// r = fl(x - fl(s~ dec(q))) quantized with its own scale (Alg. 1: base, then
// residue).  Same arithmetic per element as quant_block; the elements are
// widened one 16-byte word at a time, so only the residues are held whole.
// With an NVFP4 table (s~, fl(1/s~) of each scale byte, nv_scale_table_entry)
// the scale byte comes from nv_block_byte and s~ and the multiplier from the
// table: the same values, with a shorter dependency chain.
template <int FMT, int E, bool kResidue>
__device__ __forceinline__ void quant_block_raw(const uint4 (&raw)[E / 8], const NvScaleConst& k, uint32_t& sf,
                                                uint32_t (&codes)[E / 8], uint32_t& sfr, uint32_t (&rcodes)[E / 8],
                                                const float2* tab = nullptr) {
    auto scale = [&](float amax, float& st, float& mul) -> uint32_t {
        if (FMT == 1) return mx_block_scale(amax, st, mul);
        if (tab == nullptr) return nv_block_scale_fast(amax, k, st, mul);
        const uint32_t byte = nv_block_byte(amax, k);
        const float2 e = tab[byte];
        st = e.x;
        mul = e.y;
        return byte;
    };
    const float am = amax_bf16_words<E / 2>(reinterpret_cast<const uint32_t*>(&raw[0]));
    float st, mul;
    sf = scale(am, st, mul);
    float r[kResidue ? E : 1];
#pragma unroll
    for (int w = 0; w < E / 8; ++w) {
        const uint32_t h[4] = {raw[w].x, raw[w].y, raw[w].z, raw[w].w};
        float x[8], v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(h[i] << 16);
            x[2 * i + 1] = __uint_as_float(h[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int e = 0; e < 8; e += 2) fmul2_rn(x[e], x[e + 1], mul, mul, v[e], v[e + 1]);
        codes[w] = e2m1_encode8(v);
        if constexpr (kResidue) {
            float d[8];
            e2m1_decode8(codes[w], d);
#pragma unroll
            for (int e = 0; e < 8; ++e) r[8 * w + e] = __fsub_rn(x[e], __fmul_rn(st, d[e]));  // never fused
        }
    }
    if constexpr (kResidue) {
        float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            a0 = fmaxf(a0, fabsf(r[e]));
            a1 = fmaxf(a1, fabsf(r[e + 1]));
        }
        float rst, rmul;
        sfr = scale(fmaxf(a0, a1), rst, rmul);
#pragma unroll
        for (int w = 0; w < E / 8; ++w) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; e += 2) fmul2_rn(r[8 * w + e], r[8 * w + e + 1], rmul, rmul, v[e], v[e + 1]);
            rcodes[w] = e2m1_encode8(v);
        }
    }
}

// Eight bf16 values (one 16-byte word) widened to fp32.
__device__ __forceinline__ void unpack8_bf16(const uint4& v, float (&xf)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xf[2 * i] = __uint_as_float(w[i] << 16);
        xf[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// The 16-byte word at p, or zeros when !valid.
__device__ __forceinline__ uint4 load16_or_zero(const uint16_t* p, bool valid) {
    return valid ? *reinterpret_cast<const uint4*>(p) : make_uint4(0u, 0u, 0u, 0u);
}

// Load eight bf16 values (16 bytes) as fp32, or zeros when !valid.
__device__ __forceinline__ void load8_bf16(const uint16_t* p, bool valid, float (&xf)[8]) {
    if (valid) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xf[2 * i] = __uint_as_float(w[i] << 16);
            xf[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) xf[e] = 0.0f;
    }
}

// Byte offset of code byte b (0..127) of row r (0..127) in a 128-row x
// 128-byte tile stored in the 128-byte-swizzled shared-memory image that the
// tcgen05 K-major SW128 descriptor reads: 16-byte chunk index XOR (r % 8).
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t r, uint32_t b) {
    return r * 128u + ((((b >> 4) ^ (r & 7u))) << 4) + (b & 15u);
}

}  // namespace rs
