// Block decoders: one "line" = 64 consecutive K-elements of one weight row,
// decoded to 64 bf16 values = 8 x uint4 (chunk j holds elements 8j..8j+7,
// element 8j in the low half of .x).
//
// Decode rules (bit-exact):
//   NF4   bf16_rn( f32_rn(level[c] * absmax') ),  absmax' = absmax, or
//         f32_rn(f32(absmax_q) * absmax_scale), or with an 8-bit map
//         f32_rn( f32_rn(map[absmax_q] * absmax_scale) + offset )
//   Q4_0  bf16_rn( (nib - 8) * f32(d) )   (the fp32 product is exact)
//   Q8_0  bf16_rn( q * f32(d) )           (the fp32 product is exact)
//   Q4_K  bf16_rn( f32_rn( (d sc) q - (dmin m) ) )   (products exact)
//   FP8   bf16_rn( f32_rn( e4m3(c) * scale ) )
//   NVFP4 bf16_rn( f32_rn( e2m1(c) * f32_rn( e4m3(s_blk) * scale ) ) )
//
// NF4 and Q4_0 have 16 possible values per block: the block's 16 decoded
// bf16 values are computed once (16 fp32 multiplies + 8 conversions) and split
// into a low-byte and a high-byte plane of 16 bytes each (4 registers each).
// Each 4-bit code then picks its two bytes with byte permutes (prmt), so the
// per-element work is about two integer ops and no memory lookup.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace qlora {

// NormalFloat-4 levels as fp32 (16 standard-normal quantiles incl. an exact
// zero, divided by the largest).
__device__ __forceinline__ float nf4_level(int c) {
  switch (c) {
    case 0: return -1.0f;
    case 1: return -0.6961928f;
    case 2: return -0.52507293f;
    case 3: return -0.39491743f;
    case 4: return -0.28444132f;
    case 5: return -0.1847734f;
    case 6: return -0.09104998f;
    case 7: return 0.0f;
    case 8: return 0.079580314f;
    case 9: return 0.16093014f;
    case 10: return 0.24611226f;
    case 11: return 0.33791512f;
    case 12: return 0.44070974f;
    case 13: return 0.5626169f;
    case 14: return 0.72295666f;
    default: return 1.0f;
  }
}

// 16-entry byte-plane table of one block.
struct Lut16 {
  uint32_t lo[4];  // low bytes of entries 0..15
  uint32_t hi[4];  // high bytes of entries 0..15
};

// pairs[i] = bf16(v[2i]) | bf16(v[2i+1]) << 16
__device__ __forceinline__ Lut16 lut_from_pairs(const uint32_t (&pairs)[8]) {
  Lut16 t;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.lo[i] = prmt(pairs[2 * i], pairs[2 * i + 1], 0x6420);
    t.hi[i] = prmt(pairs[2 * i], pairs[2 * i + 1], 0x7531);
  }
  return t;
}

__device__ __forceinline__ Lut16 lut_nf4(float amax) {
  uint32_t pairs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = __fmul_rn(nf4_level(2 * i), amax);
    float b = __fmul_rn(nf4_level(2 * i + 1), amax);
    pairs[i] = pack_bf16x2(a, b);
  }
  return lut_from_pairs(pairs);
}

__device__ __forceinline__ Lut16 lut_q4_0(float d) {
  uint32_t pairs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a = __fmul_rn((float)(2 * i - 8), d);
    float b = __fmul_rn((float)(2 * i + 1 - 8), d);
    pairs[i] = pack_bf16x2(a, b);
  }
  return lut_from_pairs(pairs);
}

// Look up the 8 codes held in the 8 nibbles of w.  For the 4 codes of half h
// (nibbles 4h .. 4h+3), byte i of L[h] / H[h] receives the low / high byte of
// entry (code i).  Each half takes 4 byte permutes to fetch the candidates
// from entries 0..7 and 8..15 (selected by a code's low 3 bits) and 2 more to
// keep, per byte, the candidate its top bit names; the selectors of both
// halves come from one mask and one shift of the whole word.
__device__ __forceinline__ void lut_lookup8(const Lut16& t, uint32_t w, uint32_t (&L)[2], uint32_t (&H)[2]) {
  const uint32_t idx = w & 0x77777777u;                          // low 3 bits of each code
  const uint32_t pick = ((w >> 1) & 0x44444444u) | 0x32103210u;  // byte i of a (code < 8) or of b
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sel = h ? (idx >> 16) : idx;  // prmt reads the low 16 bits of its selector
    const uint32_t sel2 = h ? (pick >> 16) : pick;
    const uint32_t la = prmt(t.lo[0], t.lo[1], sel);
    const uint32_t lb = prmt(t.lo[2], t.lo[3], sel);
    const uint32_t ha = prmt(t.hi[0], t.hi[1], sel);
    const uint32_t hb = prmt(t.hi[2], t.hi[3], sel);
    L[h] = prmt(la, lb, sel2);
    H[h] = prmt(ha, hb, sel2);
  }
}

// ---------------------------------------------------------------- NF4 -------
// codes: 32 bytes (64 codes, element 2j in the high nibble of byte j).
__device__ __forceinline__ void decode_nf4_line(const uint4 c0, const uint4 c1, float amax, uint4 (&out)[8]) {
  const Lut16 t = lut_nf4(amax);
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t L[2], H[2], r[4];
    lut_lookup8(t, w[j], L, H);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // byte order of L/H: e(4h+1), e(4h+0), e(4h+3), e(4h+2)
      r[2 * h + 0] = prmt(L[h], H[h], 0x4051);  // elements 4h+0, 4h+1
      r[2 * h + 1] = prmt(L[h], H[h], 0x6273);  // elements 4h+2, 4h+3
    }
    out[j] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// ---------------------------------------------------------------- Q4_0 ------
// words: the 36 bytes of two consecutive 18-byte blocks (4-byte aligned).
__device__ __forceinline__ void decode_q4_0_block(uint32_t d_bits, const uint32_t (&qs)[4], uint4* out4) {
  const float d = __half2float(__ushort_as_half((unsigned short)(d_bits & 0xFFFFu)));
  const Lut16 t = lut_q4_0(d);
  uint32_t lowp[8], highp[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t L[2], H[2];
    lut_lookup8(t, qs[q], L, H);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // byte order: e(4q+2h), e(16+4q+2h), e(4q+2h+1), e(16+4q+2h+1)
      lowp[2 * q + h] = prmt(L[h], H[h], 0x6240);
      highp[2 * q + h] = prmt(L[h], H[h], 0x7351);
    }
  }
  out4[0] = make_uint4(lowp[0], lowp[1], lowp[2], lowp[3]);
  out4[1] = make_uint4(lowp[4], lowp[5], lowp[6], lowp[7]);
  out4[2] = make_uint4(highp[0], highp[1], highp[2], highp[3]);
  out4[3] = make_uint4(highp[4], highp[5], highp[6], highp[7]);
}

__device__ __forceinline__ void decode_q4_0_line(const uint32_t (&W)[9], uint4 (&out)[8]) {
  uint32_t qs0[4], qs1[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    qs0[q] = prmt(W[q], W[q + 1], 0x5432);  // bytes 2+4q .. 5+4q
    qs1[q] = W[5 + q];                      // bytes 20+4q .. 23+4q
  }
  decode_q4_0_block(W[0], qs0, &out[0]);
  decode_q4_0_block(W[4] >> 16, qs1, &out[4]);
}

// ---------------------------------------------------------------- Q8_0 ------
// Four int8 in one word -> two bf16x2 words.  int -> float by the magic
// number 2^23: float bits 0x4B0000uu = 8388608 + uu, exact for bytes.
__device__ __forceinline__ void decode_q8_word(uint32_t q, float d, uint32_t& r0, uint32_t& r1) {
  const uint32_t u = q ^ 0x80808080u;  // q + 128 as unsigned bytes
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[i] = __uint_as_float(prmt(u, 0x4B000000u, 0x7440u + i)) - 8388736.0f;  // exact: q
    f[i] = __fmul_rn(f[i], d);                                            // exact product
  }
  r0 = pack_bf16x2(f[0], f[1]);
  r1 = pack_bf16x2(f[2], f[3]);
}

__device__ __forceinline__ void decode_q8_0_block(uint32_t d_bits, const uint32_t (&qw)[8], uint4* out4) {
  const float d = __half2float(__ushort_as_half((unsigned short)(d_bits & 0xFFFFu)));
  uint32_t r[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) decode_q8_word(qw[j], d, r[2 * j], r[2 * j + 1]);
#pragma unroll
  for (int c = 0; c < 4; ++c) out4[c] = make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
}

// words: the 68 bytes of two consecutive 34-byte blocks (4-byte aligned).
__device__ __forceinline__ void decode_q8_0_line(const uint32_t (&W)[17], uint4 (&out)[8]) {
  uint32_t q0[8], q1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    q0[j] = prmt(W[j], W[j + 1], 0x5432);  // bytes 2+4j .. 5+4j
    q1[j] = W[9 + j];                      // bytes 36+4j .. 39+4j
  }
  decode_q8_0_block(W[0], q0, &out[0]);
  decode_q8_0_block(W[8] >> 16, q1, &out[4]);
}

// ---------------------------------------------------------------- FP8 -------
// Four E4M3 codes (one word, first code in the low byte) -> two bf16x2 words:
// exact conversion to fp16 and fp32, times the tensor scale (one fp32
// rounding), then bf16.
__device__ __forceinline__ void decode_fp8_word(uint32_t w, float s, uint32_t& r0, uint32_t& r1) {
  const uint32_t a = cvt_e4m3x2_f16x2(w & 0xFFFFu), b = cvt_e4m3x2_f16x2(w >> 16);
  const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a));
  const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
  r0 = pack_bf16x2(__fmul_rn(fa.x, s), __fmul_rn(fa.y, s));
  r1 = pack_bf16x2(__fmul_rn(fb.x, s), __fmul_rn(fb.y, s));
}

// words: the line's 64 codes (16 words)
__device__ __forceinline__ void decode_fp8_line(const uint32_t (&W)[17], float s, uint4 (&out)[8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t r[4];
    decode_fp8_word(W[2 * q], s, r[0], r[1]);
    decode_fp8_word(W[2 * q + 1], s, r[2], r[3]);
    out[q] = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

// -------------------------------------------------------------- NVFP4 -------
// 16-entry table of one 16-element block from its factor b = f32_rn(e4m3 block
// scale * tensor scale): codes 0..7 are the E2M1 magnitudes 0, 0.5, 1, 1.5,
// 2, 3, 4, 6 times b (each product rounded to fp32), codes 8..15 the same
// values with the sign flipped (exact).
__device__ __forceinline__ Lut16 lut_nvfp4(float b) {
  const uint32_t p0 = pack_bf16x2(__fmul_rn(0.0f, b), __fmul_rn(0.5f, b));
  const uint32_t p1 = pack_bf16x2(b, __fmul_rn(1.5f, b));
  const uint32_t p2 = pack_bf16x2(__fmul_rn(2.0f, b), __fmul_rn(3.0f, b));
  const uint32_t p3 = pack_bf16x2(__fmul_rn(4.0f, b), __fmul_rn(6.0f, b));
  Lut16 t;
  t.lo[0] = prmt(p0, p1, 0x6420);
  t.hi[0] = prmt(p0, p1, 0x7531);
  t.lo[1] = prmt(p2, p3, 0x6420);
  t.hi[1] = prmt(p2, p3, 0x7531);
  t.lo[2] = t.lo[0];
  t.lo[3] = t.lo[1];
  t.hi[2] = t.hi[0] ^ 0x80808080u;
  t.hi[3] = t.hi[1] ^ 0x80808080u;
  return t;
}

// codes: 32 bytes (64 codes, element 2j in the LOW nibble of byte j); sc4:
// the line's four E4M3 block scales (block k in byte k); ts: tensor scale.
__device__ __forceinline__ void decode_nvfp4_line(const uint32_t (&W)[17], uint32_t sc4, float ts,
                                                  uint4 (&out)[8]) {
  const uint32_t s01 = cvt_e4m3x2_f16x2(sc4 & 0xFFFFu), s23 = cvt_e4m3x2_f16x2(sc4 >> 16);
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&s01));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&s23));
  const float bs[4] = {f01.x, f01.y, f23.x, f23.y};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const Lut16 t = lut_nvfp4(__fmul_rn(bs[k], ts));
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = 2 * k + jj;  // word j: elements 8j .. 8j+7, nibble i = element 8j + i
      uint32_t L[2], H[2];
      lut_lookup8(t, W[j], L, H);
      out[j] = make_uint4(prmt(L[0], H[0], 0x5140), prmt(L[0], H[0], 0x7362), prmt(L[1], H[1], 0x5140),
                          prmt(L[1], H[1], 0x7362));
    }
  }
}

// --------------------------------------------------------------- Q4_K -------
// Scale and min of sub-block j from the 12 packed bytes s[0..2] of a
// super-block: j < 4 takes the low 6 bits of bytes j and j+4; j >= 4 takes
// byte j+4's low / high nibble and the top 2 bits of bytes j-4 / j.
__device__ __forceinline__ void q4_k_sub(const uint32_t (&s)[3], int j, int& sc, int& m) {
  auto byte = [&](int i) -> int { return (int)((s[i >> 2] >> (8 * (i & 3))) & 0xFFu); };
  if (j < 4) {
    sc = byte(j) & 63;
    m = byte(j + 4) & 63;
  } else {
    sc = (byte(j + 4) & 15) | ((byte(j - 4) >> 6) << 4);
    m = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
  }
}

// 16 entries dsc * q - dm (the product is exact, so the fused form rounds
// exactly as the product followed by the difference)
__device__ __forceinline__ Lut16 lut_q4_k(float dsc, float dm) {
  uint32_t pairs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    pairs[i] = pack_bf16x2(__fmaf_rn(dsc, (float)(2 * i), -dm), __fmaf_rn(dsc, (float)(2 * i + 1), -dm));
  return lut_from_pairs(pairs);
}

// Eight codes of one nibble plane, arranged so that nibble 2i holds element i
// and nibble 2i+1 element 4+i of the eight, decoded to four bf16x2 words in
// element order.
__device__ __forceinline__ uint4 q4_k_eight(const Lut16& t, uint32_t codes) {
  uint32_t L[2], H[2];
  lut_lookup8(t, codes, L, H);
  // half h, byte i: elements 2h, 4+2h, 2h+1, 5+2h
  return make_uint4(prmt(L[0], H[0], 0x6240), prmt(L[1], H[1], 0x6240), prmt(L[0], H[0], 0x7351),
                    prmt(L[1], H[1], 0x7351));
}

// W[0..7]: the chunk's 32 code bytes (low nibbles: sub-block 2c, elements
// 0..31; high nibbles: sub-block 2c+1, elements 32..63); W[8..11]: the
// super-block's header (fp16 d, fp16 dmin, 12 scale bytes); c: the chunk.
__device__ __forceinline__ void decode_q4_k_line(const uint32_t (&W)[17], int c, uint4 (&out)[8]) {
  const float d = __half2float(__ushort_as_half((unsigned short)(W[8] & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(W[8] >> 16)));
  const uint32_t s[3] = {W[9], W[10], W[11]};
  int sc0, m0, sc1, m1;
  q4_k_sub(s, 2 * c, sc0, m0);
  q4_k_sub(s, 2 * c + 1, sc1, m1);
  const Lut16 t0 = lut_q4_k(__fmul_rn(d, (float)sc0), __fmul_rn(dmin, (float)m0));
  const Lut16 t1 = lut_q4_k(__fmul_rn(d, (float)sc1), __fmul_rn(dmin, (float)m1));
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t a = W[2 * q], b = W[2 * q + 1];
    out[q] = q4_k_eight(t0, (a & 0x0F0F0F0Fu) | ((b & 0x0F0F0F0Fu) << 4));
    out[q + 4] = q4_k_eight(t1, ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u));
  }
}

// ------------------------------------------------- raw line loads -------------
// Where line L (= row * K/64 + kb) of each format lives.
struct WeightView {
  const uint8_t* data;
  const float* absmax;
  const int8_t* absmax_q;
  const float* absmax_scale;
  const float* amap;      // NF4: 8-bit absmax map (256 entries), or null
  const float* tscale;    // FP8 / NVFP4: the tensor's scale (one fp32)
  const uint8_t* bscale;  // NVFP4: E4M3 block scales, one byte per 16 elements
  float aoff;             // NF4 with a map: offset added to every absmax
  int dq_group;
  int dq_shift;   // log2(dq_group) when it is a power of two, else -1
  int aq_align8;  // absmax_q is 8-byte aligned
  int fmt;
};

// Raw bytes of one line, kept in registers between load and decode so the
// loads of later lines can be in flight while this one is decoded.  Nothing
// here depends on a loaded value: the NF4 absmax' = q * scale2 product is
// formed at decode time, so issuing the loads never waits for them.
constexpr int32_t kNoDq = 0x7fffffff;
struct RawLine {
  uint32_t w[17];
  float scale;  // NF4: absmax (fp32 absmax) or the group's scale2 (double
                // quantised); FP8 / NVFP4: the tensor scale
  int32_t q;    // NF4: the absmax code (double quantised), else kNoDq;
                // Q4_K: the line's chunk of its super-block
};

// NF4 absmax of the line: the fp32 absmax, RN_f32(f32(q8) * scale2), or with
// an 8-bit map RN_f32(RN_f32(map[q] * scale2) + offset)
__device__ __forceinline__ float nf4_line_scale(const RawLine& r, const WeightView& v) {
  if (r.q == kNoDq) return r.scale;
  if (v.amap != nullptr) return __fadd_rn(__fmul_rn(__ldg(v.amap + (r.q & 0xFF)), r.scale), v.aoff);
  return __fmul_rn((float)r.q, r.scale);
}

enum { FMT_BF16 = 0, FMT_NF4 = 1, FMT_Q8_0 = 2, FMT_Q4_0 = 3, FMT_Q4_K = 4, FMT_FP8 = 5, FMT_NVFP4 = 6 };

template <int FMT>
__device__ __forceinline__ void load_line(const WeightView& v, int64_t line, RawLine& r) {
  if constexpr (FMT == FMT_NF4) {
    const uint4 a = ldg_nc_v4(v.data + line * 32);
    const uint4 b = ldg_nc_v4(v.data + line * 32 + 16);
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
    if (v.absmax != nullptr) {
      r.scale = __ldg(v.absmax + line);
      r.q = kNoDq;
    } else {
      r.q = (int32_t)__ldg(v.absmax_q + line);
      const int64_t grp = v.dq_shift >= 0 ? (line >> v.dq_shift) : line / v.dq_group;
      r.scale = __ldg(v.absmax_scale + grp);
    }
  } else if constexpr (FMT == FMT_Q8_0 || FMT == FMT_Q4_0) {
    // 68- or 36-byte lines of a 16-byte aligned array: a line starts 8-byte
    // aligned when its index is even and is 8-byte aligned from its second
    // word otherwise, so it takes 8-byte loads and one 4-byte load
    constexpr int WORDS = FMT == FMT_Q8_0 ? 17 : 9;
    const uint8_t* p = v.data + line * (4 * WORDS);
    if ((line & 1) == 0) {
#pragma unroll
      for (int i = 0; i < WORDS / 2; ++i) {
        const uint2 w = ldg_nc_v2(p + 8 * i);
        r.w[2 * i] = w.x;
        r.w[2 * i + 1] = w.y;
      }
      r.w[WORDS - 1] = ldg_nc_u32(p + 4 * (WORDS - 1));
    } else {
      r.w[0] = ldg_nc_u32(p);
#pragma unroll
      for (int i = 0; i < WORDS / 2; ++i) {
        const uint2 w = ldg_nc_v2(p + 4 + 8 * i);
        r.w[1 + 2 * i] = w.x;
        r.w[2 + 2 * i] = w.y;
      }
    }
  } else if constexpr (FMT == FMT_FP8) {  // 64 code bytes
    const uint4* p = reinterpret_cast<const uint4*>(v.data + line * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = ldg_nc_v4(p + i);
      r.w[4 * i] = a.x; r.w[4 * i + 1] = a.y; r.w[4 * i + 2] = a.z; r.w[4 * i + 3] = a.w;
    }
    r.scale = __ldg(v.tscale);
  } else if constexpr (FMT == FMT_NVFP4) {  // 32 code bytes + 4 block scales
    const uint4 a = ldg_nc_v4(v.data + line * 32);
    const uint4 b = ldg_nc_v4(v.data + line * 32 + 16);
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
    r.w[8] = ldg_nc_u32(v.bscale + line * 4);
    r.scale = __ldg(v.tscale);
  } else if constexpr (FMT == FMT_Q4_K) {  // chunk (line & 3) of 144-byte super-block (line >> 2)
    const uint8_t* sb = v.data + (line >> 2) * 144;
    const uint4 h = ldg_nc_v4(sb);
    const uint4 a = ldg_nc_v4(sb + 16 + (line & 3) * 32);
    const uint4 b = ldg_nc_v4(sb + 32 + (line & 3) * 32);
    r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
    r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
    r.w[8] = h.x; r.w[9] = h.y; r.w[10] = h.z; r.w[11] = h.w;
    r.q = (int32_t)(line & 3);
  } else {  // BF16: 128 bytes
    const uint4* p = reinterpret_cast<const uint4*>(v.data + line * 128);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = ldg_nc_v4(p + i);
      r.w[4 * i] = a.x; r.w[4 * i + 1] = a.y; r.w[4 * i + 2] = a.z; r.w[4 * i + 3] = a.w;
    }
  }
}

// NF4: the line's absmax fields only (its code bytes arrive another way).
__device__ __forceinline__ void load_nf4_scale(const WeightView& v, int64_t line, RawLine& r) {
  if (v.absmax != nullptr) {
    r.scale = __ldg(v.absmax + line);
    r.q = kNoDq;
  } else {
    r.q = (int32_t)__ldg(v.absmax_q + line);
    const int64_t grp = v.dq_shift >= 0 ? (line >> v.dq_shift) : line / v.dq_group;
    r.scale = __ldg(v.absmax_scale + grp);
  }
}

// The fields of a line that do not come with its code bytes (the code bytes
// arrive through a shared-memory ring): NF4 absmax, FP8 / NVFP4 tensor scale,
// NVFP4 block scales, Q4_K chunk index.
template <int FMT>
__device__ __forceinline__ void load_line_side(const WeightView& v, int64_t line, RawLine& r) {
  if constexpr (FMT == FMT_NF4) {
    load_nf4_scale(v, line, r);
  } else if constexpr (FMT == FMT_FP8) {
    r.scale = __ldg(v.tscale);
  } else if constexpr (FMT == FMT_NVFP4) {
    r.w[8] = ldg_nc_u32(v.bscale + line * 4);
    r.scale = __ldg(v.tscale);
  } else if constexpr (FMT == FMT_Q4_K) {
    r.q = (int32_t)(line & 3);
  }
}

// Only for the quantised formats.
template <int FMT>
__device__ __forceinline__ void decode_line(const RawLine& r, const WeightView& v, uint4 (&out)[8]) {
  if constexpr (FMT == FMT_NF4) {
    decode_nf4_line(make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]), make_uint4(r.w[4], r.w[5], r.w[6], r.w[7]),
                    nf4_line_scale(r, v), out);
  } else if constexpr (FMT == FMT_FP8) {
    decode_fp8_line(r.w, r.scale, out);
  } else if constexpr (FMT == FMT_NVFP4) {
    decode_nvfp4_line(r.w, r.w[8], r.scale, out);
  } else if constexpr (FMT == FMT_Q4_K) {
    decode_q4_k_line(r.w, r.q, out);
  } else if constexpr (FMT == FMT_Q8_0) {
    uint32_t W[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) W[i] = r.w[i];
    decode_q8_0_line(W, out);
  } else if constexpr (FMT == FMT_Q4_0) {
    uint32_t W[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) W[i] = r.w[i];
    decode_q4_0_line(W, out);
  }
}

}  // namespace qlora
