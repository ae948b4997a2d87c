// Steps a1-a3 of the path: amax reduction, fp32 scale, RNE cast to FP8.
//
// Definitions ("fp8_parity.py", scaled_roundtrip): s = (amax / fmax) clamped
// below at 1e-12, byte = (x / s).to(fp8).  The quotient must be the correctly
// rounded fp32 division.  Per scale we form r = RN(1/s) once and, per element,
//   q0 = RN(x r);  e = x - q0 s (exact, one FMA);  q = RN(q0 + e r)
// which is Markstein's correction step (P. Markstein, IBM J. Res. Dev. 34(1),
// 1990; Muller et al., Handbook of Floating-Point Arithmetic, ch. on
// division): with r within half an ulp of 1/s it returns RN(x / s) whenever
// the remainder does not underflow.  Here s >= 1e-12, so a remainder can only
// underflow for |x / s| < 2^-63, where every FP8 code is a signed zero; the
// sign is restored with copysign.  The correction is only used on data whose
// quotients stay below the FP8 overflow point (checked per thread, row,
// column or block from the amax already at hand); anything else -- Inf or NaN
// scales or data, overflowing quotients -- takes true IEEE division and the
// explicit NaN / Inf / saturation rules.
//
// Kernel layout: one CTA of 256 threads owns a 128x128 input tile at a time
// (grid-stride over tiles).  Thread (warp w, lane l) holds rows
// [8 rg, 8 rg + 8) and columns [8 cg, 8 cg + 8) of the tile with
// rg = 2 w + l / 16, cg = l % 16: eight 16-byte loads, each warp instruction
// covering two full 256-byte row segments (bf16).  Row amax for 1x128 tiles
// is a shuffle butterfly inside each half-warp; column amax for 128x1 tiles
// goes through shared memory; the transposed FP8 copy is an in-register 8x8
// byte transpose (uniform scales) or a second cast (column-tile scales).
//
// MXFP8 (the "mxfp8" recipe; the pages give no encoding, so the OCP
// Microscaling Formats v1.0 specification defines it): blocks of 32 elements
// share an E8M0 scale X = 2^(floor(log2 amax) - emax_elem); the biased
// exponent of amax's fp32 bit pattern gives that directly, X is a power of
// two, and the element is the saturating conversion of the exact product
// x * (1 / X): no division is involved.
#include <cuda.h>
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fp8q_internal.h"
#include "fp8q_ptx.cuh"

namespace fp8q {
namespace {

constexpr int kQuantThreads = 256;

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<FP8Q_E4M3> {
  static constexpr float kMax = 448.0f;
  static constexpr float kFastLimit = 460.0f;  // below the 464 overflow midpoint
  static constexpr __nv_fp8_interpretation_t kInterp = __NV_E4M3;
};
template <>
struct FmtTraits<FP8Q_E5M2> {
  static constexpr float kMax = 57344.0f;
  static constexpr float kFastLimit = 61000.0f;  // below the 61440 midpoint
  static constexpr __nv_fp8_interpretation_t kInterp = __NV_E5M2;
};

__device__ __forceinline__ uint32_t abs_bits(float v) {
  return __float_as_uint(v) & 0x7FFFFFFFu;
}

// s = max(fl32(amax / fmax), fl32(1e-12)); a NaN amax gives a NaN scale.
__device__ __forceinline__ float scale_from_amax(float amax, float fm) {
  float s = __fdiv_rn(amax, fm);
  return (s < 1e-12f) ? 1e-12f : s;
}

// Two fp32 values -> two FP8 bytes (lo in the low byte), RNE, saturating.
template <int FMT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                             FmtTraits<FMT>::kInterp);
}

// Two fp32 values (x -> low byte, y -> high byte) -> two FP8 bytes.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_pair(float2 v) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, FmtTraits<FMT>::kInterp);
}

// Correctly rounded x / s for a pair, packed two-wide (see the file comment;
// nsn = (-s, -s), r2 = (r, r)).  Signs of zero results are fixed by the caller.
__device__ __forceinline__ float2 div2_fast(float2 x, float2 nsn, float2 r2) {
  const float2 q0 = __fmul2_rn(x, r2);
  const float2 e = __ffma2_rn(q0, nsn, x);
  return __ffma2_rn(e, r2, q0);
}

// Full-rule encode for the slow path: NaN -> 0x7F | sign; without saturation
// an overflowing quotient becomes NaN (E4M3) or Inf (E5M2).
template <int FMT>
__device__ __forceinline__ uint32_t encode_slow(float v, int saturate) {
  uint32_t sgn = (__float_as_uint(v) >> 24) & 0x80u;
  if (v != v) return 0x7Fu | sgn;
  if (!saturate) {
    float a = fabsf(v);
    if (FMT == FP8Q_E4M3) {
      if (a > 464.0f) return 0x7Fu | sgn;
    } else {
      if (a >= 61440.0f) return 0x7Cu | sgn;
    }
  }
  return cvt2<FMT>(v, 0.0f) & 0xFFu;
}

template <int FMT>
__device__ __forceinline__ uint2 cast8_fast(const float (&v)[8], float s, float r) {
  const float2 nsn = make_float2(-s, -s), r2 = make_float2(r, r);
  uint32_t p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 q = div2_fast(make_float2(v[2 * k], v[2 * k + 1]), nsn, r2);
    q.x = copysignf(q.x, v[2 * k]);       // a zero quotient keeps x's sign
    q.y = copysignf(q.y, v[2 * k + 1]);
    p[k] = cvt_pair<FMT>(q);
  }
  return make_uint2(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410));
}

// Slow path per element: a NaN input keeps its sign (0x7F | sign); a NaN the
// division creates (NaN scale, Inf / Inf) is 0x7F; everything else is the
// IEEE quotient under the full encode rules.
template <int FMT>
__device__ __forceinline__ uint32_t cast1_slow(float x, float s, int saturate) {
  if (x != x) return 0x7Fu | ((__float_as_uint(x) >> 24) & 0x80u);
  const float v = __fdiv_rn(x, s);
  if (v != v) return 0x7Fu;
  return encode_slow<FMT>(v, saturate);
}

// Out of line, with the eight values as scalars: they travel in registers,
// so a caller's fast path keeps no copy of them in local memory.
template <int FMT>
__device__ __noinline__ uint2 cast8_slow(float v0, float v1, float v2, float v3, float v4,
                                         float v5, float v6, float v7, float s, int saturate) {
  const uint32_t b0 = cast1_slow<FMT>(v0, s, saturate), b1 = cast1_slow<FMT>(v1, s, saturate);
  const uint32_t b2 = cast1_slow<FMT>(v2, s, saturate), b3 = cast1_slow<FMT>(v3, s, saturate);
  const uint32_t b4 = cast1_slow<FMT>(v4, s, saturate), b5 = cast1_slow<FMT>(v5, s, saturate);
  const uint32_t b6 = cast1_slow<FMT>(v6, s, saturate), b7 = cast1_slow<FMT>(v7, s, saturate);
  return make_uint2(b0 | (b1 << 8) | (b2 << 16) | (b3 << 24),
                    b4 | (b5 << 8) | (b6 << 16) | (b7 << 24));
}

template <int FMT>
__device__ __forceinline__ uint2 cast8(const float (&v)[8], float s, float r, bool fast,
                                       int saturate) {
  if (fast) return cast8_fast<FMT>(v, s, r);
  return cast8_slow<FMT>(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], s, saturate);
}

// Quotients of every value with |x| <= m stay on the fast path's domain.
template <int FMT>
__device__ __forceinline__ bool fast_ok(uint32_t m_bits, float r) {
  return (r > 0.0f) && (__uint_as_float(m_bits) * r <= FmtTraits<FMT>::kFastLimit);
}

// Eight consecutive input elements of one row, kept in their storage type
// (bf16 stays packed two to a register).  at(j) widens element j to fp32.
template <typename InT>
struct Row8;

template <>
struct Row8<uint16_t> {
  uint4 w;
  __device__ __forceinline__ void load(const void *base, int64_t idx) {
    w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + idx));
  }
  __device__ __forceinline__ void zero() { w = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void load_smem(const uint8_t *row_base) {
    w = *reinterpret_cast<const uint4 *>(row_base);
  }
  __device__ __forceinline__ uint32_t word(int k) const {
    return k == 0 ? w.x : (k == 1 ? w.y : (k == 2 ? w.z : w.w));
  }
  __device__ __forceinline__ float at(int j) const {
    const uint32_t x = word(j >> 1);
    return (j & 1) ? __uint_as_float(x & 0xFFFF0000u) : __uint_as_float(x << 16);
  }
  // max |element| as an fp32 bit pattern
  __device__ __forceinline__ uint32_t absmax_bits() const {
    const uint32_t k = 0x7FFF7FFFu;
    const uint32_t m = __vmaxu2(__vmaxu2(w.x & k, w.y & k), __vmaxu2(w.z & k, w.w & k));
    return max(m & 0xFFFFu, m >> 16) << 16;
  }
  // per-column running max |x|, packed: cm[k] holds columns 2k, 2k+1
  static constexpr int kColWords = 4;
  __device__ __forceinline__ void colmax_update(uint32_t (&cm)[kColWords]) const {
    const uint32_t k = 0x7FFF7FFFu;
    cm[0] = __vmaxu2(cm[0], w.x & k);
    cm[1] = __vmaxu2(cm[1], w.y & k);
    cm[2] = __vmaxu2(cm[2], w.z & k);
    cm[3] = __vmaxu2(cm[3], w.w & k);
  }
  __device__ __forceinline__ static uint32_t colmax_bits(const uint32_t (&cm)[kColWords], int j) {
    const uint32_t x = cm[j >> 1];
    return (j & 1) ? (x & 0xFFFF0000u) : (x << 16);
  }
};

template <>
struct Row8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const void *base, int64_t idx) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx);
    a = __ldg(p);
    b = __ldg(p + 1);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void load_smem(const uint8_t *row_base) {
    const float4 *q = reinterpret_cast<const float4 *>(row_base);
    a = q[0];
    b = q[1];
  }
  __device__ __forceinline__ float at(int j) const {
    switch (j) {
      case 0: return a.x; case 1: return a.y; case 2: return a.z; case 3: return a.w;
      case 4: return b.x; case 5: return b.y; case 6: return b.z; default: return b.w;
    }
  }
  __device__ __forceinline__ uint32_t absmax_bits() const {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, abs_bits(at(j)));
    return m;
  }
  static constexpr int kColWords = 8;
  __device__ __forceinline__ void colmax_update(uint32_t (&cm)[kColWords]) const {
#pragma unroll
    for (int j = 0; j < 8; ++j) cm[j] = max(cm[j], abs_bits(at(j)));
  }
  __device__ __forceinline__ static uint32_t colmax_bits(const uint32_t (&cm)[kColWords], int j) {
    return cm[j];
  }
};

// Fast cast of one 8-element bf16 row chunk straight from its packed words:
// pairs are widened, divided two-wide and converted two at a time; the FP8
// sign bits are then OR-ed in from the bf16 sign bits (bit 7 of bytes 1 and
// 3 of each word), which is exact for every finite x (a negative x always
// has a negative code, -0 included) and fixes zero quotients.
template <int FMT>
__device__ __forceinline__ uint2 cast_row_fast(const Row8<uint16_t> &x, float s, float r) {
  const float2 nsn = make_float2(-s, -s), r2 = make_float2(r, r);
  uint32_t p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = x.word(k);
    p[k] = cvt_pair<FMT>(div2_fast(
        make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), nsn, r2));
  }
  const uint32_t lo = __byte_perm(p[0], p[1], 0x5410) |
                      (__byte_perm(x.w.x, x.w.y, 0x7531) & 0x80808080u);
  const uint32_t hi = __byte_perm(p[2], p[3], 0x5410) |
                      (__byte_perm(x.w.z, x.w.w, 0x7531) & 0x80808080u);
  return make_uint2(lo, hi);
}

template <int FMT>
__device__ __forceinline__ uint2 cast_row_fast(const Row8<float> &x, float s, float r) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = x.at(j);
  return cast8_fast<FMT>(v, s, r);
}

template <int FMT, typename InT>
__device__ __forceinline__ uint2 cast_row(const Row8<InT> &x, float s, float r, bool fast,
                                          int saturate) {
  if (fast) return cast_row_fast<FMT>(x, s, r);
  return cast8_slow<FMT>(x.at(0), x.at(1), x.at(2), x.at(3), x.at(4), x.at(5), x.at(6),
                         x.at(7), s, saturate);
}

// ------------------------------------------------------------------ MXFP8

// E8M0 code of a block from the fp32 bit pattern of its max |x|.  For a
// normal max, floor(log2 amax) = E - 127 with E the biased exponent, so the
// shared exponent floor(log2 amax) - emax_elem is E - 127 - emax_elem and its
// E8M0 code (bias 127) is E - emax_elem; a zero or subnormal max (E = 0), or
// any code below E8M0's range, clamps to 0 (2^-127); an Inf or NaN max gives
// the NaN code 0xFF.  emax_elem: 448 = 1.75 * 2^8, 57344 = 1.75 * 2^15.
template <int FMT>
__device__ __forceinline__ uint32_t mx_code(uint32_t amax_bits) {
  constexpr int kEmax = FMT == FP8Q_E4M3 ? 8 : 15;
  const int e = (int)(amax_bits >> 23);
  if (e == 255) return 0xFFu;
  return (uint32_t)max(e - kEmax, 0);
}

// 1 / X = 2^(127 - code) for a finite code (0..254): 2^-127 is subnormal.
__device__ __forceinline__ float mx_inv_scale(uint32_t code) {
  return code >= 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - code) << 23);
}

// Eight elements times 1/X (exact), saturating RNE to FP8; the sign bits are
// OR-ed in from the inputs so that a negative value that rounds to zero is
// -0 (0x80).  A NaN block (code 0xFF) writes 0x7F everywhere.
template <int FMT>
__device__ __forceinline__ uint2 mx_cast_row(const Row8<uint16_t> &x, uint32_t code) {
  if (code == 0xFFu) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const float f = mx_inv_scale(code);
  const float2 f2 = make_float2(f, f);
  uint32_t p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w = x.word(k);
    p[k] = cvt_pair<FMT>(
        __fmul2_rn(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), f2));
  }
  const uint32_t lo = __byte_perm(p[0], p[1], 0x5410) |
                      (__byte_perm(x.w.x, x.w.y, 0x7531) & 0x80808080u);
  const uint32_t hi = __byte_perm(p[2], p[3], 0x5410) |
                      (__byte_perm(x.w.z, x.w.w, 0x7531) & 0x80808080u);
  return make_uint2(lo, hi);
}

template <int FMT>
__device__ __forceinline__ uint2 mx_cast8(const float (&v)[8], uint32_t code) {
  if (code == 0xFFu) return make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  const float f = mx_inv_scale(code);
  const float2 f2 = make_float2(f, f);
  uint32_t p[4], sg[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    p[k] = cvt_pair<FMT>(__fmul2_rn(make_float2(v[2 * k], v[2 * k + 1]), f2));
#pragma unroll
  for (int j = 0; j < 8; ++j)
    sg[j >> 2] |= ((__float_as_uint(v[j]) >> 31) << 7) << (8 * (j & 3));
  return make_uint2(__byte_perm(p[0], p[1], 0x5410) | sg[0],
                    __byte_perm(p[2], p[3], 0x5410) | sg[1]);
}

template <int FMT>
__device__ __forceinline__ uint2 mx_cast_row(const Row8<float> &x, uint32_t code) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = x.at(j);
  return mx_cast8<FMT>(v, code);
}

// Byte offset, inside a tile's 512-byte scale atom, of the scale of row r
// (0..127 of the tile) and 32-wide K block j (0..3): the layout the GEMM's
// tensor memory copy (32 rows of 16 bytes, replicated over the four lane
// quarters) turns into what the block-scaled MMA reads.
__device__ __forceinline__ int mx_atom_offset(int r, int j) {
  return (r & 31) * 16 + (r >> 5) * 4 + j;
}

// 4x4 byte transpose: a..d are rows (byte k = column k); o0..o3 are columns.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t &o0, uint32_t &o1, uint32_t &o2,
                                             uint32_t &o3) {
  uint32_t t0 = __byte_perm(a, b, 0x5140);
  uint32_t t1 = __byte_perm(a, b, 0x7362);
  uint32_t t2 = __byte_perm(c, d, 0x5140);
  uint32_t t3 = __byte_perm(c, d, 0x7362);
  o0 = __byte_perm(t0, t2, 0x5410);
  o1 = __byte_perm(t0, t2, 0x7632);
  o2 = __byte_perm(t1, t3, 0x5410);
  o3 = __byte_perm(t1, t3, 0x7632);
}

// rows[i] holds row i (8 bytes, columns 0..7); cols[j] receives column j.
__device__ __forceinline__ void transpose8x8(const uint2 (&rows)[8], uint2 (&cols)[8]) {
  transpose4x4(rows[0].x, rows[1].x, rows[2].x, rows[3].x, cols[0].x, cols[1].x, cols[2].x,
               cols[3].x);
  transpose4x4(rows[4].x, rows[5].x, rows[6].x, rows[7].x, cols[0].y, cols[1].y, cols[2].y,
               cols[3].y);
  transpose4x4(rows[0].y, rows[1].y, rows[2].y, rows[3].y, cols[4].x, cols[5].x, cols[6].x,
               cols[7].x);
  transpose4x4(rows[4].y, rows[5].y, rows[6].y, rows[7].y, cols[4].y, cols[5].y, cols[6].y,
               cols[7].y);
}

// Kernel variants.
enum KernelMode : int {
  kKTensor = 0,     // uniform scale from a device amax
  kKDelayed = 1,    // uniform scale from the history, amax pushed after
  kKTileRow = 2,    // 1x128 row tiles -> q, q_scales
  kKTileCol = 3,    // 128x1 column tiles -> q_t, qt_scales
  kKTileBoth = 4,   // both from one read
  kKBlock = 5,      // 128x128 blocks -> q and/or q_t, block scales
  kKRowAmax = 6,    // row-wise pass 1: per-row / per-column amax, atomicMax into
                    // q_scales / qt_scales (as fp32 bit patterns)
  kKRowCast = 7,    // row-wise pass 2: cast with the scales of those amaxes
  kKTensorFused = 8, // per-tensor current scaling in one cooperative launch:
                     // amax over every tile, a grid barrier, then the cast
  kKMx = 9           // MXFP8: 1x32 row blocks -> q and/or 32x1 column blocks
                     // -> q_t, each with its tile's 512-byte E8M0 atom
};

// Dynamic tile scheduling: each launch of the quantize kernel takes one slot
// (round-robin over kQuantWorkSlots, so launches that overlap in time use
// different slots); work[0] hands out tile indices, work[1] counts CTAs that
// are done, and the last CTA returns both to zero for the slot's next launch.
constexpr int kQuantWorkSlots = 256;
__device__ unsigned int g_quant_work[2 * kQuantWorkSlots];

// Input tiles (128 x 128 elements) reach shared memory by TMA through a ring
// of kStages buffers; thread 0 claims the next tile and refills a buffer as
// soon as every thread has copied its part of the previous tile out of it, so
// up to kStages tiles per CTA are in flight while earlier ones are converted
// and stored.  Claiming tiles as CTAs free up (rather than a fixed stride)
// evens out SMs that stream at different rates.
template <typename InT>
struct QuantRing {
  static constexpr int kTileBytes = 128 * 128 * (int)sizeof(InT);
  static constexpr int kStages = sizeof(InT) == 2 ? 3 : 2;
};

// CTAs per SM a mode is built for: bf16 input runs three CTAs of two-stage
// rings (the same tiles in flight per SM as two CTAs of three stages, with 50%
// more warps to hide the cast's latency; every mode fits 85 registers without
// spills), except the column-tile modes, whose scratch plus the 8 KB
// transposed-copy staging leave room for two CTAs of three stages; fp32 input
// keeps its two-stage ring of 64 KB tiles.
template <typename InT, int KM>
struct QuantShape {
  // modes that can write the transposed copy stage it through shared memory
  static constexpr bool kStaging = !(KM == kKTileRow || KM == kKRowAmax);
  static constexpr int kStageBytes = kStaging ? 64 * 128 : 0;
  // the column-tile modes' own scratch would not leave room for three
  static constexpr bool kThree = sizeof(InT) == 2 && !(KM == kKTileCol || KM == kKTileBoth ||
                                                       KM == kKRowCast || KM == kKMx);
  static constexpr int kMinBlocks = kThree ? 3 : 2;
  static constexpr int kStages = kThree ? 2 : QuantRing<InT>::kStages;
  static constexpr int kTileBytes = QuantRing<InT>::kTileBytes;
  // MXFP8: the tile's two 512-byte scale atoms are assembled in shared memory
  static constexpr int kMxBytes = KM == kKMx ? 1024 : 0;
  static constexpr int kSmemBytes = kStages * kTileBytes + kStageBytes + kMxBytes + 1024;
};

template <typename InT, int FMT, int KM>
__global__ void __launch_bounds__(kQuantThreads, (QuantShape<InT, KM>::kMinBlocks))
    quant2d_kernel(const __grid_constant__ CUtensorMap tmx, const QuantParams p) {
  constexpr bool kRowTiles = (KM == kKTileRow || KM == kKTileBoth);
  constexpr bool kColTiles = (KM == kKTileCol || KM == kKTileBoth);
  constexpr bool kRowwise = (KM == kKRowAmax || KM == kKRowCast);
  constexpr bool kFused = (KM == kKTensorFused);
  constexpr bool kUniform = (KM == kKTensor || KM == kKDelayed || KM == kKBlock || kFused);
  constexpr bool kMx = (KM == kKMx);
  using Ring = QuantShape<InT, KM>;
  const float fm = FmtTraits<FMT>::kMax;

  extern __shared__ uint8_t dyn_smem[];
  __shared__ float sh_row_s[128], sh_row_r[128];
  __shared__ float sh_col_s[128], sh_col_r[128];
  __shared__ uint32_t sh_colmax[8][128];
  __shared__ uint32_t sh_red[8];
  __shared__ __align__(8) uint64_t sh_full[Ring::kStages];
  __shared__ int sh_tr[Ring::kStages], sh_tc[Ring::kStages];  // tile of a stage; -1: none
  __shared__ int sh_abort;
  __shared__ uint32_t sh_amax_bits;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp * 2 + (lane >> 4);
  const int cg = lane & 15;
  const int64_t rows = p.rows, cols = p.cols;
  const int64_t tiles_c = (cols + 127) / 128, tiles_r = (rows + 127) / 128;
  const int64_t ntiles = tiles_r * tiles_c;
  const int saturate = p.saturate;
  const uint32_t raw = ptx::smem_u32(dyn_smem);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint8_t *ring_ptr = dyn_smem + (ring - raw);
  uint8_t *qt_stage = dyn_smem + (ring - raw) + Ring::kStages * Ring::kTileBytes;
  uint8_t *mx_stage = qt_stage + Ring::kStageBytes;   // MX: rows atom, then columns atom
  volatile int *abort_flag = &sh_abort;

  // The transposed FP8 tile (q_t rows c0.., byte columns r0..) goes out as
  // whole 128-byte rows: each thread's 8 x 8 bytes (cb[j] = q_t row
  // cbase + j, bytes rbase..rbase+7) are staged in shared memory, 64 q_t rows
  // at a time, then 8 consecutive threads write one row.  The 16-byte chunk
  // of a row is XOR-swizzled by its 8-row group so that the staging writes of
  // a warp hit distinct banks.  Every thread of the CTA must call this.
  auto store_qt = [&](const uint2 (&cb)[8], bool valid, int64_t r0, int64_t c0) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      if (valid && (cg >> 3) == half) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int row = (cg & 7) * 8 + j;
          const int chunk = (rg >> 1) ^ (cg & 7);
          *reinterpret_cast<uint2 *>(qt_stage + row * 128 + chunk * 16 + (rg & 1) * 8) = cb[j];
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = tid + k * kQuantThreads;
        const int row = c >> 3, chunk = c & 7;
        const int64_t qrow = c0 + half * 64 + row;   // input column
        const int64_t qcol = r0 + chunk * 16;          // input row (rows % 16 == 0)
        if (qrow < cols && qcol < rows)
          *reinterpret_cast<uint4 *>(p.q_t + qrow * rows + qcol) =
              *reinterpret_cast<const uint4 *>(qt_stage + row * 128 +
                                               (chunk ^ ((row >> 3) & 7)) * 16);
      }
      __syncthreads();
    }
  };

  // Per-tensor current scaling runs right after the amax pass over the same
  // data, so it hands out the tiles backwards and meets the most recently read
  // (still L2-resident) part of x first.
  unsigned int *work = &g_quant_work[2 * p.work_slot];
  unsigned int next_claim = 0;  // thread 0: claimed, not yet issued
  // Work order: a CTA's first kStages tiles are blockIdx.x + j * gridDim.x
  // (loaded at once).  With p.dynamic every later tile is claimed from the
  // slot's counter, numbered on from kStages * gridDim.x; otherwise the fixed
  // stride continues (few tiles per CTA leave little tail to even out, and
  // the claims' cost would show).
  // thread 0: start the load of pipeline step i for tile number c; a step past
  // the last tile carries -1 and completes with no data.  Claims are made one
  // step ahead of their use, so the atomic's round trip overlaps a tile's
  // work.  One CTA's tile numbers only grow (one thread's claims on one
  // address come back in increasing order), so after a -1 every later step
  // is -1 as well.
  // Fused per-tensor mode: a CTA's T tiles are blockIdx.x + j * gridDim.x;
  // steps 0..T-1 take the amax over them, steps T..2T-1 cast them in reverse
  // order (the most recently read, likeliest still in L2, first).
  const int64_t my_tiles =
      (blockIdx.x < ntiles) ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto fused_tile = [&](int64_t i) -> int64_t {
    if (i < my_tiles) return (int64_t)blockIdx.x + i * gridDim.x;
    if (i < 2 * my_tiles) return (int64_t)blockIdx.x + (2 * my_tiles - 1 - i) * gridDim.x;
    return ntiles;
  };
  auto issue_tile = [&](int64_t i, int64_t c) {
    const int s = (int)(i % Ring::kStages);
    const uint32_t bar = ptx::smem_u32(&sh_full[s]);
    if (c < ntiles) {
      const int64_t t = (KM == kKTensor) ? ntiles - 1 - c : c;
      const int tr = (int)(t / tiles_c);
      const int tc = (int)(t - (int64_t)tr * tiles_c);
      sh_tr[s] = tr;
      sh_tc[s] = tc;
      ptx::mbar_arrive_expect_tx(bar, Ring::kTileBytes);
      ptx::tma_load_2d(ring + s * Ring::kTileBytes, &tmx, tc * 128, tr * 128, bar);
    } else {
      sh_tr[s] = -1;
      ptx::mbar_arrive(bar);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < Ring::kStages; ++s) ptx::mbar_init(ptx::smem_u32(&sh_full[s]), 1);
    sh_abort = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&tmx);
#pragma unroll
    for (int j = 0; j < Ring::kStages; ++j)
      issue_tile(j, kFused ? fused_tile(j) : (int64_t)blockIdx.x + (int64_t)j * gridDim.x);
    if (p.dynamic) next_claim = atomicAdd(&work[0], 1u);
  }
  __syncthreads();

  float s_u = 0.0f, r_u = 0.0f;
  if (KM == kKTensor) {
    s_u = scale_from_amax(*p.amax_in, fm);
    r_u = __fdiv_rn(1.0f, s_u);
  } else if (KM == kKDelayed) {
    uint32_t h = 0;
#pragma unroll
    for (int i = 0; i < FP8Q_HISTORY_LEN; ++i) h = max(h, abs_bits(p.hist->amax[i]));
    s_u = scale_from_amax(__uint_as_float(h), fm);
    r_u = __fdiv_rn(1.0f, s_u);
  }
  uint32_t run_max = 0;  // delayed: running max |x| of this CTA
  int64_t issued = Ring::kStages;  // thread 0's count of claimed pipeline steps

  // Every thread takes every iteration's barriers; the loop ends for all
  // threads at once (a CTA-wide abort verdict, or a stage without a tile).
  for (int64_t i = 0;; ++i) {
    const int s = (int)(i % Ring::kStages);
    const uint32_t parity = (uint32_t)((i / Ring::kStages) & 1);
    const bool ok = ptx::wait_bounded_warp(ptx::smem_u32(&sh_full[s]), parity, abort_flag, p.err);
    const int tr = ok ? *reinterpret_cast<volatile int *>(&sh_tr[s]) : -1;
    const int tc = ok ? *reinterpret_cast<volatile int *>(&sh_tc[s]) : 0;
    const int64_t r0 = (int64_t)tr * 128, c0 = (int64_t)tc * 128;
    const int64_t cbase = c0 + cg * 8;
    const int64_t rbase = r0 + rg * 8;
    const bool col_ok = cbase < cols;
    const bool rchunk_ok = rbase < rows;

    // Copy this thread's 8 x 8 block out of the staged tile (row-major,
    // 128 elements per row; out-of-bounds rows and columns were zero-filled).
    Row8<InT> v[8];
    const uint8_t *tile_ptr = ring_ptr + s * Ring::kTileBytes;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      if (ok && tr >= 0) v[r].load_smem(tile_ptr + ((rg * 8 + r) * 128 + cg * 8) * (int)sizeof(InT));
      else v[r].zero();
    }
    // One CTA-wide verdict, so every thread leaves the loop at the same
    // iteration; this barrier also frees buffer s.  All threads read the same
    // stage tile, so `tr < 0` is uniform too.
    const bool all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (!all_ok || tr < 0) break;
    if (tid == 0 && !*abort_flag) {
      if (kFused) {
        issue_tile(i + Ring::kStages, fused_tile(i + Ring::kStages));
      } else if (p.dynamic) {
        issue_tile(i + Ring::kStages, (int64_t)Ring::kStages * gridDim.x + next_claim);
        next_claim = atomicAdd(&work[0], 1u);
      } else {
        issue_tile(i + Ring::kStages, (int64_t)blockIdx.x + (i + Ring::kStages) * gridDim.x);
      }
      issued = i + Ring::kStages + 1;
    }

    if (kFused && i == my_tiles) {
      // Every CTA has taken the amax of its tiles: publish, wait for all the
      // others (bounded), then every CTA reads the tensor's amax.
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, run_max);
      if (lane == 0) sh_red[warp] = m;
      __syncthreads();
      if (tid == 0) {
        uint32_t cm = sh_red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) cm = max(cm, sh_red[w]);
        unsigned int *amax_bits = reinterpret_cast<unsigned int *>(p.amax_out);
        if (cm != 0) atomicMax(amax_bits, cm);
        __threadfence();
        atomicAdd(&work[0], 1u);
        const uint64_t t0 = ptx::globaltimer_ns();
        while (*reinterpret_cast<volatile unsigned int *>(&work[0]) < gridDim.x) {
          if (ptx::globaltimer_ns() - t0 > ptx::kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.err, 1u);
            break;
          }
          __nanosleep(64);
        }
        __threadfence();
        sh_amax_bits = *reinterpret_cast<volatile unsigned int *>(amax_bits);
      }
      __syncthreads();
      s_u = scale_from_amax(__uint_as_float(sh_amax_bits), fm);
      r_u = __fdiv_rn(1.0f, s_u);
    }

    uint32_t rowmax[8];
    uint32_t cmp[Row8<InT>::kColWords];
    uint32_t tmax = 0;
    if (kRowTiles || kUniform || kRowwise || kMx) {
#pragma unroll
      for (int i = 0; i < 8; ++i) rowmax[i] = v[i].absmax_bits();
    }
    if (kColTiles || kRowwise || kMx) {
#pragma unroll
      for (int k = 0; k < Row8<InT>::kColWords; ++k) cmp[k] = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i].colmax_update(cmp);
    }
    if (kUniform) {
#pragma unroll
      for (int i = 0; i < 8; ++i) tmax = max(tmax, rowmax[i]);
    }

    // ------------------------------------------------ uniform-scale modes
    if (kFused && i < my_tiles) {
      run_max = max(run_max, tmax);   // amax pass: nothing is stored
    } else if (kUniform) {
      float s = s_u, r = r_u;
      if (KM == kKBlock) {
        uint32_t m = __reduce_max_sync(0xFFFFFFFFu, tmax);
        if (lane == 0) sh_red[warp] = m;
        __syncthreads();
        uint32_t bm = sh_red[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) bm = max(bm, sh_red[w]);
        s = scale_from_amax(__uint_as_float(bm), fm);
        r = __fdiv_rn(1.0f, s);
        if (tid == 0) p.q_scales[tr * tiles_c + tc] = s;
      }
      if (KM == kKDelayed) run_max = max(run_max, tmax);
      const bool fast = fast_ok<FMT>(tmax, r);
      uint2 rb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) rb[i] = cast_row<FMT>(v[i], s, r, fast, saturate);
      if (p.q != nullptr && col_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (rbase + i < rows)
            *reinterpret_cast<uint2 *>(p.q + (rbase + i) * cols + cbase) = rb[i];
      }
      if (p.q_t != nullptr) {
        uint2 cb[8];
        transpose8x8(rb, cb);
        store_qt(cb, col_ok && rchunk_ok, r0, c0);
      }
    }

    // ------------------------------------------------------ 1x128 row tiles
    if (kRowTiles) {
      // Butterfly over the 16 lanes of a half-warp that share these 8 rows:
      // each exchange halves the rows a lane keeps, so 8 shuffles reduce all
      // 8 rows.  Afterwards lanes cg and cg^1 hold the max of row
      // rsel = 4 b3 + 2 b2 + b1 (b_k = bit k of cg).
      const bool h3 = cg & 8, h2 = cg & 4, h1 = cg & 2;
      uint32_t a4[4];
#pragma unroll
      for (int t4 = 0; t4 < 4; ++t4) {
        uint32_t keep = h3 ? rowmax[t4 + 4] : rowmax[t4];
        uint32_t send = h3 ? rowmax[t4] : rowmax[t4 + 4];
        a4[t4] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
      }
      uint32_t a2[2];
#pragma unroll
      for (int t2 = 0; t2 < 2; ++t2) {
        uint32_t keep = h2 ? a4[t2 + 2] : a4[t2];
        uint32_t send = h2 ? a4[t2] : a4[t2 + 2];
        a2[t2] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
      }
      uint32_t a1 = max(h1 ? a2[1] : a2[0], __shfl_xor_sync(0xFFFFFFFFu, h1 ? a2[0] : a2[1], 2));
      a1 = max(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 1));
      const int rsel = (h3 ? 4 : 0) + (h2 ? 2 : 0) + (h1 ? 1 : 0);
      if ((cg & 1) == 0) {
        float s = scale_from_amax(__uint_as_float(a1), fm);
        sh_row_s[rg * 8 + rsel] = s;
        sh_row_r[rg * 8 + rsel] = __fdiv_rn(1.0f, s);
        if (rbase + rsel < rows) p.q_scales[tc * rows + rbase + rsel] = s;
      }
      __syncwarp();
      if (col_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float s = sh_row_s[rg * 8 + i], r = sh_row_r[rg * 8 + i];
          uint2 b = cast_row<FMT>(v[i], s, r, fast_ok<FMT>(rowmax[i], r), saturate);
          if (rbase + i < rows) *reinterpret_cast<uint2 *>(p.q + (rbase + i) * cols + cbase) = b;
        }
      }
    }

    // --------------------------------------------------- 128x1 column tiles
    if (kColTiles) {
      uint32_t colmax[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        colmax[j] = Row8<InT>::colmax_bits(cmp, j);
        colmax[j] = max(colmax[j], __shfl_xor_sync(0xFFFFFFFFu, colmax[j], 16));
      }
      if (lane < 16) {
        *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8]) =
            make_uint4(colmax[0], colmax[1], colmax[2], colmax[3]);
        *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8 + 4]) =
            make_uint4(colmax[4], colmax[5], colmax[6], colmax[7]);
      }
      __syncthreads();
      if (tid < 128) {
        uint32_t m = sh_colmax[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) m = max(m, sh_colmax[w][tid]);
        float s = scale_from_amax(__uint_as_float(m), fm);
        sh_col_s[tid] = s;
        sh_col_r[tid] = __fdiv_rn(1.0f, s);
        if (c0 + tid < cols) p.qt_scales[tr * cols + c0 + tid] = s;
      }
      __syncthreads();
      uint2 cb[8];
      const bool valid = col_ok && rchunk_ok;
      if (valid) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float s = sh_col_s[cg * 8 + j], r = sh_col_r[cg * 8 + j];
          float cv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) cv[i] = v[i].at(j);
          cb[j] = cast8<FMT>(cv, s, r, fast_ok<FMT>(colmax[j], r), saturate);
        }
      }
      store_qt(cb, valid, r0, c0);
    }
    // ------------------------------------------- row-wise scaling, pass 1
    if (KM == kKRowAmax) {
      if (p.q_scales != nullptr) {
        // same half-warp butterfly as the 1x128 rows, then one atomicMax per row
        const bool h3 = cg & 8, h2 = cg & 4, h1 = cg & 2;
        uint32_t a4[4];
#pragma unroll
        for (int t4 = 0; t4 < 4; ++t4) {
          uint32_t keep = h3 ? rowmax[t4 + 4] : rowmax[t4];
          uint32_t send = h3 ? rowmax[t4] : rowmax[t4 + 4];
          a4[t4] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 8));
        }
        uint32_t a2[2];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          uint32_t keep = h2 ? a4[t2 + 2] : a4[t2];
          uint32_t send = h2 ? a4[t2] : a4[t2 + 2];
          a2[t2] = max(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 4));
        }
        uint32_t a1 = max(h1 ? a2[1] : a2[0], __shfl_xor_sync(0xFFFFFFFFu, h1 ? a2[0] : a2[1], 2));
        a1 = max(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 1));
        const int rsel = (h3 ? 4 : 0) + (h2 ? 2 : 0) + (h1 ? 1 : 0);
        if ((cg & 1) == 0 && rbase + rsel < rows)
          atomicMax(reinterpret_cast<unsigned int *>(p.q_scales) + rbase + rsel, a1);
      }
      if (p.qt_scales != nullptr) {
        uint32_t colmax[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          colmax[j] = Row8<InT>::colmax_bits(cmp, j);
          colmax[j] = max(colmax[j], __shfl_xor_sync(0xFFFFFFFFu, colmax[j], 16));
        }
        if (lane < 16) {
          *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8]) =
              make_uint4(colmax[0], colmax[1], colmax[2], colmax[3]);
          *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8 + 4]) =
              make_uint4(colmax[4], colmax[5], colmax[6], colmax[7]);
        }
        __syncthreads();
        if (tid < 128 && c0 + tid < cols) {
          uint32_t m = sh_colmax[0][tid];
#pragma unroll
          for (int w = 1; w < 8; ++w) m = max(m, sh_colmax[w][tid]);
          atomicMax(reinterpret_cast<unsigned int *>(p.qt_scales) + c0 + tid, m);
        }
      }
    }

    // ------------------------------------------- row-wise scaling, pass 2
    if (KM == kKRowCast) {
      // scales of this tile's 128 rows / 128 columns from the pass-1 amaxes
      if (tid < 128) {
        if (p.q_scales != nullptr) {
          const float a = (r0 + tid < rows) ? p.q_scales[r0 + tid] : 0.0f;
          const float sr = scale_from_amax(a, fm);
          sh_row_s[tid] = sr;
          sh_row_r[tid] = __fdiv_rn(1.0f, sr);
        }
        if (p.qt_scales != nullptr) {
          const float a = (c0 + tid < cols) ? p.qt_scales[c0 + tid] : 0.0f;
          const float sc = scale_from_amax(a, fm);
          sh_col_s[tid] = sc;
          sh_col_r[tid] = __fdiv_rn(1.0f, sc);
        }
      }
      __syncthreads();
      if (p.q_scales != nullptr && col_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float sr = sh_row_s[rg * 8 + i], rr = sh_row_r[rg * 8 + i];
          uint2 b = cast_row<FMT>(v[i], sr, rr, fast_ok<FMT>(rowmax[i], rr), saturate);
          if (rbase + i < rows) *reinterpret_cast<uint2 *>(p.q + (rbase + i) * cols + cbase) = b;
        }
      }
      if (p.qt_scales != nullptr) {
        uint2 cb[8];
        const bool valid = col_ok && rchunk_ok;
        if (valid) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float sc = sh_col_s[cg * 8 + j], rc = sh_col_r[cg * 8 + j];
            float cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cv[i] = v[i].at(j);
            cb[j] = cast8<FMT>(cv, sc, rc,
                               fast_ok<FMT>(Row8<InT>::colmax_bits(cmp, j), rc), saturate);
          }
        }
        store_qt(cb, valid, r0, c0);
      }
    }
    // -------------------------------------------------------------- MXFP8
    if (kMx) {
      if (p.q != nullptr) {
        // 1x32 row blocks: the four lanes cg = 4 b .. 4 b + 3 of a half-warp
        // hold one block of each of their 8 rows
        const int jblk = cg >> 2;
        uint32_t code[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t m = max(rowmax[i], __shfl_xor_sync(0xFFFFFFFFu, rowmax[i], 1));
          m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
          code[i] = mx_code<FMT>(m);
        }
        if ((cg & 3) == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) mx_stage[mx_atom_offset(rg * 8 + i, jblk)] = (uint8_t)code[i];
        }
        if (col_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint2 b = mx_cast_row<FMT>(v[i], code[i]);
            if (rbase + i < rows) *reinterpret_cast<uint2 *>(p.q + (rbase + i) * cols + cbase) = b;
          }
        }
      }
      if (p.q_t != nullptr) {
        // 32x1 column blocks: rows 32 t .. 32 t + 31 of the tile belong to
        // warps 2 t and 2 t + 1 (both half-warps of each)
        uint32_t colmax[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          colmax[j] = Row8<InT>::colmax_bits(cmp, j);
          colmax[j] = max(colmax[j], __shfl_xor_sync(0xFFFFFFFFu, colmax[j], 16));
        }
        if (lane < 16) {
          *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8]) =
              make_uint4(colmax[0], colmax[1], colmax[2], colmax[3]);
          *reinterpret_cast<uint4 *>(&sh_colmax[warp][cg * 8 + 4]) =
              make_uint4(colmax[4], colmax[5], colmax[6], colmax[7]);
        }
        __syncthreads();
        const int wpair = warp & ~1;
        uint32_t ccode[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ccode[j] = mx_code<FMT>(max(sh_colmax[wpair][cg * 8 + j], sh_colmax[wpair + 1][cg * 8 + j]));
        if ((warp & 1) == 0 && lane < 16) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            mx_stage[512 + mx_atom_offset(cg * 8 + j, warp >> 1)] = (uint8_t)ccode[j];
        }
        uint2 cb[8];
        const bool valid = col_ok && rchunk_ok;
        if (valid) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) cv[i] = v[i].at(j);
            cb[j] = mx_cast8<FMT>(cv, ccode[j]);
          }
        }
        store_qt(cb, valid, r0, c0);
      }
      __syncthreads();   // the tile's atoms are complete
      if (p.q != nullptr && tid < 32)
        reinterpret_cast<uint4 *>(p.mx_scales + ((int64_t)tr * tiles_c + tc) * 512)[tid] =
            reinterpret_cast<const uint4 *>(mx_stage)[tid];
      if (p.q_t != nullptr && tid >= 32 && tid < 64)
        reinterpret_cast<uint4 *>(p.mxt_scales + ((int64_t)tc * tiles_r + tr) * 512)[tid - 32] =
            reinterpret_cast<const uint4 *>(mx_stage + 512)[tid - 32];
    }

    // Shared scratch that crosses warps is reused by the next tile.  Per-tensor,
    // delayed and 1x128 row-tile casts keep theirs per warp (ordered by the
    // barrier at the top of the next iteration).
    if (!(KM == kKTensor || KM == kKDelayed || KM == kKTileRow || kFused)) __syncthreads();
  }

  if (tid == 0) {
    if (*abort_flag) {
      // Let copies still in flight land before the CTA exits (bounded).
      for (int64_t j = (issued > Ring::kStages ? issued - Ring::kStages : 0); j < issued; ++j) {
        const uint32_t bar = ptx::smem_u32(&sh_full[j % Ring::kStages]);
        const uint32_t par = (uint32_t)((j / Ring::kStages) & 1);
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, par) && ptx::globaltimer_ns() - t0 < 200000000ull) {
        }
      }
    }
    // Every claim of this CTA precedes its "done"; the last CTA resets the slot.
    const bool uses_slot = p.dynamic || kFused;
    if (uses_slot) __threadfence();
    if (uses_slot && atomicAdd(&work[1], 1u) == gridDim.x - 1) {
      work[0] = 0u;
      work[1] = 0u;
      __threadfence();
    }
  }

  // ------------------------------------------ per-tensor scale bookkeeping
  if (KM == kKTensor || kFused) {
    if (blockIdx.x == 0 && tid == 0 && p.scale_out != nullptr) *p.scale_out = s_u;
  }
  if (KM == kKDelayed) {
    uint32_t m = __reduce_max_sync(0xFFFFFFFFu, run_max);
    if (lane == 0) sh_red[warp] = m;
    __syncthreads();
    if (tid == 0) {
      uint32_t cm = sh_red[0];
#pragma unroll
      for (int w = 1; w < 8; ++w) cm = max(cm, sh_red[w]);
      fp8q_amax_history *h = p.hist;
      atomicMax(&h->pending, cm);
      __threadfence();
      const unsigned prev = atomicAdd(&h->arrivals, 1u);
      if (prev == gridDim.x - 1) {
        // Last CTA: every other CTA has read the history and published its
        // amax.  Push the tensor's amax into the ring and reset the scratch.
        __threadfence();
        const uint32_t amax_bits = atomicExch(&h->pending, 0u);
        const int nx = h->next;
        h->amax[nx] = __uint_as_float(amax_bits);
        h->next = (nx + 1) % FP8Q_HISTORY_LEN;
        h->scale = s_u;
        if (p.scale_out != nullptr) *p.scale_out = s_u;
        __threadfence();
        atomicExch(&h->arrivals, 0u);
      }
    }
  }
}

// amax over a flat array: 16-byte loads, packed 16-bit max for bf16,
// warp/CTA reduction; each CTA stores its maximum (as an fp32 bit pattern:
// |x| bit patterns order like the values, NaN patterns above Inf) in its own
// entry of a slot of g_amax_partials and takes a ticket, and the last CTA
// reduces the partials with all its threads and writes the output.  The call
// therefore needs no zeroing launch ahead of it, and no two CTAs contend on
// one address except for the ticket.  Each launch takes its own slot
// (round-robin), so launches that overlap in time do not share one.
constexpr int kAmaxSlots = 32;
constexpr int kAmaxMaxCtas = 8 * 256;   // partial entries per slot (grids of <= 8 CTAs per SM)
__device__ unsigned int g_amax_partials[kAmaxSlots][kAmaxMaxCtas];
__device__ unsigned int g_amax_tickets[kAmaxSlots];

// Each CTA streams 32 KB chunks of x (chunk c = blockIdx.x + k gridDim.x)
// through a ring of kAmaxStages shared-memory stages filled by bulk copies
// (cp.async.bulk, completion counted on one mbarrier per stage); all 256
// threads reduce each chunk from shared memory.  Bulk copies keep far more
// bytes in flight per SM than per-thread 16-byte loads can.  The bytes after
// the last whole chunk are read with plain loads.
constexpr int kAmaxChunk = 32768;
constexpr int kAmaxStages = 6;
constexpr int kAmaxSmem = kAmaxStages * kAmaxChunk + 128;

template <typename InT>
__global__ void __launch_bounds__(256, 1)
    amax_kernel(const InT *__restrict__ x, int64_t n, unsigned int *out, int slot,
                unsigned int *err) {
  extern __shared__ uint8_t amax_smem[];
  __shared__ __align__(8) uint64_t bars[kAmaxStages];
  __shared__ uint32_t red[8];
  __shared__ int last, abort_flag;
  uint8_t *ring = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(amax_smem) + 127) & ~static_cast<uintptr_t>(127));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t nbytes = n * (int64_t)sizeof(InT);
  const int64_t nchunks = nbytes / kAmaxChunk;
  const int64_t mine = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint8_t *xb = reinterpret_cast<const uint8_t *>(x);
  auto issue = [&](int64_t j) {   // thread 0: load this CTA's j-th chunk into stage j % S
    const uint32_t bar = ptx::smem_u32(&bars[j % kAmaxStages]);
    ptx::mbar_arrive_expect_tx(bar, kAmaxChunk);
    ptx::bulk_load(ptx::smem_u32(ring + (j % kAmaxStages) * kAmaxChunk),
                   xb + (blockIdx.x + j * gridDim.x) * (int64_t)kAmaxChunk, kAmaxChunk, bar);
  };
  if (tid == 0) {
    for (int s = 0; s < kAmaxStages; ++s) ptx::mbar_init(ptx::smem_u32(&bars[s]), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
    for (int64_t j = 0; j < mine && j < kAmaxStages; ++j) issue(j);
  }
  __syncthreads();
  uint32_t m = 0;
  auto upd = [&](uint4 w) {
    if (sizeof(InT) == 2) {
      m = __vmaxu2(m, w.x & 0x7FFF7FFFu);
      m = __vmaxu2(m, w.y & 0x7FFF7FFFu);
      m = __vmaxu2(m, w.z & 0x7FFF7FFFu);
      m = __vmaxu2(m, w.w & 0x7FFF7FFFu);
    } else {
      m = max(m, w.x & 0x7FFFFFFFu);
      m = max(m, w.y & 0x7FFFFFFFu);
      m = max(m, w.z & 0x7FFFFFFFu);
      m = max(m, w.w & 0x7FFFFFFFu);
    }
  };
  int64_t issued = mine < kAmaxStages ? mine : kAmaxStages;
  for (int64_t j = 0; j < mine; ++j) {
    const int s = (int)(j % kAmaxStages);
    const bool ok = ptx::wait_bounded_warp(ptx::smem_u32(&bars[s]),
                                           (uint32_t)((j / kAmaxStages) & 1), &abort_flag, err);
    if (ok) {
      const uint4 *st = reinterpret_cast<const uint4 *>(ring + s * kAmaxChunk);
#pragma unroll
      for (int k = 0; k < kAmaxChunk / 16 / 256; ++k) upd(st[tid + k * 256]);
    }
    // every thread is done with stage s (or the CTA is aborting): refill it
    if (__syncthreads_or(ok ? 0 : 1)) break;
    if (tid == 0 && j + kAmaxStages < mine) {
      issue(j + kAmaxStages);
      issued = j + kAmaxStages + 1;
    }
  }
  if (tid == 0 && abort_flag) {
    // let the copies in flight land before the CTA exits (bounded)
    for (int64_t j = issued > kAmaxStages ? issued - kAmaxStages : 0; j < issued; ++j) {
      const uint64_t t0 = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(ptx::smem_u32(&bars[j % kAmaxStages]),
                                 (uint32_t)((j / kAmaxStages) & 1)) &&
             ptx::globaltimer_ns() - t0 < 200000000ull) {
      }
    }
  }
  // the bytes after the last whole chunk, with plain loads
  const int64_t tail0 = nchunks * kAmaxChunk;
  const int64_t nvec_tail = (nbytes - tail0) / 16;
  const uint4 *tv = reinterpret_cast<const uint4 *>(xb + tail0);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + tid; i < nvec_tail;
       i += (int64_t)gridDim.x * blockDim.x)
    upd(__ldg(tv + i));
  if (sizeof(InT) == 2) m = max(m & 0xFFFFu, m >> 16) << 16;
  // the elements after the last whole 16 bytes
  const int64_t first_scalar = (tail0 + nvec_tail * 16) / (int64_t)sizeof(InT);
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + tid;
  if (g < n - first_scalar) {
    const int64_t k = first_scalar + g;
    uint32_t b;
    if (sizeof(InT) == 2)
      b = ((uint32_t) reinterpret_cast<const uint16_t *>(x)[k] << 16) & 0x7FFFFFFFu;
    else
      b = __float_as_uint(reinterpret_cast<const float *>(x)[k]) & 0x7FFFFFFFu;
    m = max(m, b);
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  unsigned int *partials = g_amax_partials[slot];
  if (tid == 0) {
    uint32_t r = red[0];
    for (int w = 1; w < 8; ++w) r = max(r, red[w]);
    partials[blockIdx.x] = r;
    __threadfence();                                   // the partial before the ticket
    last = atomicAdd(&g_amax_tickets[slot], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  // the last CTA: every partial is visible (each was fenced before its ticket)
  __threadfence();
  uint32_t r = 0;
  for (int k = tid; k < (int)gridDim.x; k += blockDim.x)
    r = max(r, *reinterpret_cast<volatile unsigned int *>(&partials[k]));
  r = __reduce_max_sync(0xFFFFFFFFu, r);
  __syncthreads();
  if (lane == 0) red[warp] = r;
  __syncthreads();
  if (tid == 0) {
    for (int w = 0; w < 8; ++w) r = max(r, red[w]);
    *out = r;
    g_amax_tickets[slot] = 0u;
  }
}

template <typename InT, int FMT, int KM>
cudaError_t launch_variant(const QuantParams &p, cudaStream_t stream) {
  using Ring = QuantShape<InT, KM>;
  auto kernel = quant2d_kernel<InT, FMT, KM>;
  static PerDeviceOnce setup;  // per instantiation: resident CTAs per SM, 0 on failure
  const int blocks_per_sm = setup.get([&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Ring::kSmemBytes) != cudaSuccess)
      return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kQuantThreads,
                                                      Ring::kSmemBytes) != cudaSuccess)
      return 0;
    return n < 1 ? 1 : n;
  });
  if (blocks_per_sm < 1) return cudaErrorInvalidDeviceFunction;
  // The input as a 2D tensor: cols elements per row, rows rows; one box is a
  // 128 x 128 tile, out-of-bounds parts zero-filled.  rows == 0 or cols == 0
  // launches no tile and leaves the map unused.
  CUtensorMap tmx;
  memset(&tmx, 0, sizeof tmx);
  const int64_t ntiles = ((p.rows + 127) / 128) * ((p.cols + 127) / 128);
  if (ntiles > 0 &&
      !make_tmap_2d(&tmx, p.x,
                    sizeof(InT) == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                    (uint64_t)p.cols, (uint64_t)p.rows, (uint64_t)p.cols * sizeof(InT), 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (ntiles > 0x7FFFFFFF) return cudaErrorInvalidValue;  // tile indices are 32-bit
  int64_t grid = (int64_t)sm_count() * blocks_per_sm;
  if (ntiles < grid) grid = ntiles;
  if (grid < 1) grid = 1;
  static std::atomic<unsigned int> next_slot{0};
  QuantParams q = p;
  q.dynamic = (KM != kKTensorFused && ntiles >= 8 * grid) ? 1 : 0;
  q.work_slot = (q.dynamic || KM == kKTensorFused)
                    ? (int)(next_slot.fetch_add(1u) % kQuantWorkSlots)
                    : 0;
  if (log_enabled()) {
    static const char *const kModeNames[] = {"tensor",   "delayed",  "tile_rows", "tile_cols",
                                             "tile_both", "block",   "row_amax",  "row_cast",
                                             "tensor_fused", "mx"};
    fprintf(stderr,
            "[fp8q] launch quant2d_kernel mode %s %s input, %lld tiles of 128x128, grid %lld "
            "(%d per SM)%s%s\n",
            kModeNames[KM], sizeof(InT) == 2 ? "bf16" : "fp32", (long long)ntiles,
            (long long)grid, blocks_per_sm, q.dynamic ? ", tiles claimed dynamically" : "",
            KM == kKTensorFused ? ", cooperative" : "");
  }
  if (KM == kKTensorFused) {
    // every CTA must be resident for the grid barrier: a cooperative launch
    // guarantees it (or fails)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.dynamicSmemBytes = Ring::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tmx, q);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  kernel<<<(unsigned)grid, kQuantThreads, Ring::kSmemBytes, stream>>>(tmx, q);
  return cudaGetLastError();
}

template <typename InT, int FMT>
cudaError_t dispatch_mode(const QuantParams &p, cudaStream_t stream) {
  switch (p.mode) {
    case kModeTensorCurrent:
      return launch_variant<InT, FMT, kKTensor>(p, stream);
    case kModeTensorDelayed:
      return launch_variant<InT, FMT, kKDelayed>(p, stream);
    case kModeBlock:
      return launch_variant<InT, FMT, kKBlock>(p, stream);
    case kModeRowAmax:
      return launch_variant<InT, FMT, kKRowAmax>(p, stream);
    case kModeRowCast:
      return launch_variant<InT, FMT, kKRowCast>(p, stream);
    case kModeTensorFused:
      return launch_variant<InT, FMT, kKTensorFused>(p, stream);
    case kModeMx:
      return launch_variant<InT, FMT, kKMx>(p, stream);
    case kModeTile:
      if (p.q != nullptr && p.q_t != nullptr) return launch_variant<InT, FMT, kKTileBoth>(p, stream);
      if (p.q != nullptr) return launch_variant<InT, FMT, kKTileRow>(p, stream);
      return launch_variant<InT, FMT, kKTileCol>(p, stream);
  }
  return cudaErrorInvalidValue;
}

// Row-wise pass 3: the amaxes left in a scale array become scales.
__global__ void __launch_bounds__(256) amax_to_scale_kernel(float *s, int64_t n, float fm) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) s[i] = scale_from_amax(s[i], fm);
}

}  // namespace

cudaError_t launch_amax_to_scale(float *s, int64_t n, int format, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const float fm = format == FP8Q_E4M3 ? 448.0f : 57344.0f;
  amax_to_scale_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(s, n, fm);
  return cudaGetLastError();
}

cudaError_t launch_quant2d(const QuantParams &p, cudaStream_t stream) {
  if (p.in_dtype == FP8Q_DT_BF16) {
    return p.format == FP8Q_E4M3 ? dispatch_mode<uint16_t, FP8Q_E4M3>(p, stream)
                                 : dispatch_mode<uint16_t, FP8Q_E5M2>(p, stream);
  }
  return p.format == FP8Q_E4M3 ? dispatch_mode<float, FP8Q_E4M3>(p, stream)
                               : dispatch_mode<float, FP8Q_E5M2>(p, stream);
}

cudaError_t launch_amax(const void *x, int in_dtype, int64_t n, float *amax,
                        cudaStream_t stream) {
  // one CTA per SM (its ring takes 192 KB of shared memory), or one per
  // whole chunk when there are fewer; n == 0 still runs one CTA, which
  // writes 0
  const int64_t nbytes = n * (in_dtype == FP8Q_DT_BF16 ? 2 : 4);
  int64_t blocks = nbytes / kAmaxChunk;
  int64_t cap = sm_count();
  if (cap > kAmaxMaxCtas) cap = kAmaxMaxCtas;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  static std::atomic<unsigned int> next_slot{0};
  const int slot = (int)(next_slot.fetch_add(1u) % kAmaxSlots);
  unsigned int *out = reinterpret_cast<unsigned int *>(amax);
  unsigned int *err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidValue;
  static PerDeviceOnce setup[2];   // bf16, fp32 input
  const int t = in_dtype == FP8Q_DT_BF16 ? 0 : 1;
  const int ready = setup[t].get([&] {
    const cudaError_t e = t == 0 ? cudaFuncSetAttribute(amax_kernel<uint16_t>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        kAmaxSmem)
                                 : cudaFuncSetAttribute(amax_kernel<float>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        kAmaxSmem);
    return e == cudaSuccess ? 1 : 0;
  });
  if (ready != 1) return cudaErrorInvalidDeviceFunction;
  if (log_enabled())
    fprintf(stderr, "[fp8q] launch amax_kernel %s input, %lld elements, grid %lld\n",
            in_dtype == FP8Q_DT_BF16 ? "bf16" : "fp32", (long long)n, (long long)blocks);
  if (in_dtype == FP8Q_DT_BF16)
    amax_kernel<uint16_t><<<(unsigned)blocks, 256, kAmaxSmem, stream>>>(
        static_cast<const uint16_t *>(x), n, out, slot, err);
  else
    amax_kernel<float><<<(unsigned)blocks, 256, kAmaxSmem, stream>>>(
        static_cast<const float *>(x), n, out, slot, err);
  return cudaGetLastError();
}

}  // namespace fp8q
