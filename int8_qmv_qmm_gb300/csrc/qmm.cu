// qmm: fused dequantise-into-matmul on the tcgen05 tensor cores (batched
// decode and prefill).
//
// y[m][n] = sum_k x[m][k] * w_hat[n][k],  w_hat = q*scale + bias (per group of 64)
//
// The reconstructed weight only ever exists in tensor memory, as the MMA's A
// operand: it is never written to DRAM, nor to shared memory ("track(upstream-
// iree): fused dequant->matmul for the packed int8 bandwidth win", section
// "The blocker (measured)").
//
// Orientation ("swap AB"): the MMA's M dimension is 128 weight rows and its N
// dimension is a tile of BN = 16..256 tokens (a stage costs about the same
// for every N up to 256, since the issuing thread's per-stage latency, not
// the tensor pipe, sets it; so the tile may be wider than the batch, rows
// past M being zero-filled by the TMA).
//   D[n][m] (TMEM, f32) += W_hat[n][k] (TMEM, A operand) * x[m][k] (smem, B)
//
// Persistent CTAs (one per SM) walk 128 x BN output tiles, or, when the tiles
// are too few for the SMs, a cluster of 2 or 4 CTAs shares each tile, each
// CTA taking a slice of K, and the partial accumulators are summed through
// distributed shared memory at the end (by the epilogue warps and the first
// dequantising warpgroup, idle by then).  The K loop runs in stages of one
// group (64 k) through a ring of shared-memory stages and, with the same
// index, of TMEM A slots:
//   warp 0       TMA producer: x tile [BN x 64] (128-byte swizzle), packed
//                tile [128 rows x 64 codes] (32/64-byte swizzle) and, when the
//                scale rows are 16-byte aligned, the 8-group scale and bias
//                boxes holding the stage's group.
//   warp 1       TMEM allocator and MMA issuer (one thread): per stage one
//                wait, for the stage's A slot (its dequantisers waited for
//                the stage's TMA bytes first), then 4 MMAs of K=16 (A from
//                the stage's TMEM slot, B = x from shared memory) into a TMEM
//                accumulator (two, alternating by tile, when BN <= 128), and
//                tcgen05.commit to free the stage / hand the tile over.
//   warps 2..9   two dequantising warpgroups taking stages in turn (thread =
//                weight row = TMEM lane): unpack the row's 64 codes, w_hat =
//                q*scale + bias in the operand type with one fused
//                multiply-add (bit-identical to qlin_dequant's output), and
//                write the row into the stage's A slot with one tcgen05.st.
//                Keeping A out of shared memory leaves its bandwidth to the
//                TMA writes and the MMA's reads of x.
//                bfloat16 keeps only 8 significant bits, so rounding w_hat to
//                it moves a weight by up to 2^-8 of its value, as much as the
//                whole output tolerance.  For bfloat16 the A slot therefore
//                holds two operands, hi = RNE(w_hat) (the reconstruction
//                itself) and a residual lo, and each K step issues two MMAs
//                into the same accumulator: hi + lo is w_hat to about 2^-15,
//                and rounding hi + lo to bfloat16 gives back hi exactly.
//                float16 (11 bits) needs no residual.
//   warps 10..13 epilogue: tcgen05.ld of their TMEM lane quarter, the layer
//                bias if any (qlin_linear_ex), RNE to the output type (or
//                float32), stores along n; with two accumulators it overlaps
//                the next tile's K loop.
//
// Every mbarrier wait is bounded (about 2 s); a wait that gives up records a
// bit in a device status word, the CTA unwinds (waiting, bounded, for its own
// TMA copies and MMAs in flight), frees its TMEM and exits.

#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "sm100_ptx.cuh"

namespace qlin {

__device__ unsigned int g_qmm_status = 0;

namespace {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 64;           // k per stage (one group)
constexpr int kDequantGroups = 2;   // warpgroups that dequantise stages in rotation
constexpr int kDequantWarps = 4 * kDequantGroups;
constexpr int kThreads = (2 + kDequantWarps + 4) * 32;  // TMA, MMA, dequant, 4 epilogue warps

enum : unsigned {
  kStatusProducer = 1u,
  kStatusMma = 2u,
  kStatusDequant = 4u,
  kStatusEpilogue = 8u,
  kStatusTeardown = 16u,
};

__device__ __forceinline__ void report(unsigned bit) { atomicOr(&g_qmm_status, bit); }

// D (TMEM, f32) += A (TMEM: row i in lane i, K along columns, two 16-bit
// elements per 32-bit column, element k in the low half) * B (shared memory
// descriptor); M = 128, accumulate = 0 overwrites D.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Each thread of the warp writes 32 consecutive 32-bit columns of its own TMEM
// lane (lane = the warp's lane quarter * 32 + lane id, taken from taddr).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Wait until this thread's tcgen05.st have completed.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


template <int BITS>
struct Geo {
  static constexpr int kWordsPerGroup = kBK * BITS / 32;           // 8 or 16
  static constexpr int kPackedRowBytes = kWordsPerGroup * 4;       // 32 or 64
  static constexpr int kPackedBytes = kBM * kPackedRowBytes;       // 4 or 8 KB
};

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Operands per weight in the A slot: 1 (float16: w_hat), 2 (bfloat16: hi and
// the residual lo, see lo_pair).
template <typename AT>
struct OperandSplit {
  static constexpr int value = std::is_same<AT, __nv_bfloat16>::value ? 2 : 1;
};

// Shared-memory stage: [x tile][packed tile][8 groups of scales, of biases].
// TMEM: kDBufs accumulators of BN columns, then one slot of SPLIT x 32 columns
// per ring stage holding the stage's dequantised A tile(s) (128 lanes x 64
// 16-bit values each).
// BOX: the stage holds the scale and bias boxes (they come by TMA); without
// them a stage is 4 KB smaller, which can make room for one more stage.
template <int BITS, int BN, int SPLIT, bool BOX>
struct Layout {
  static constexpr int kXBytes = BN * kBK * 2;           // x tile, 128-byte rows
  static constexpr int kWBytes = Geo<BITS>::kPackedBytes;
  static constexpr int kSBytes = 2 * kBM * 16;           // 8 groups of scales + of biases
  static constexpr int kWOff = round_up(kXBytes, 1024);
  static constexpr int kSOff = kWOff + round_up(kWBytes, 1024);
  static constexpr int kStageBytes = kSOff + (BOX ? round_up(kSBytes, 1024) : 0);
  static constexpr int kTxBytes = kXBytes + kWBytes;
  // two accumulators (the epilogue of a tile overlaps the next tile's K loop)
  // unless they would leave TMEM too few A slots
  static constexpr int kDBufs = BN >= 256 ? 1 : 2;
  static constexpr int kACol0 = kDBufs * BN < 32 ? 32 : kDBufs * BN;
  static constexpr int kAColsPerStage = SPLIT * kBK / 2;  // 64 16-bit values per lane each
  static constexpr int kMaxStages = (512 - kACol0) / kAColsPerStage;
};

// ---- unpack + dequantise one 16-bit pair: returns (w_hat[2j], w_hat[2j+1])
template <typename AT>
__device__ __forceinline__ uint32_t fma_pair(uint32_t magic_pair, uint32_t s2, uint32_t b2) {
  using T2 = typename Act<AT>::T2;
  const uint32_t mq = Act<AT>::kMagic2;
  T2 v = *reinterpret_cast<const T2*>(&magic_pair);
  const T2 m = *reinterpret_cast<const T2*>(&mq);
  const T2 q = __hsub2(v, m);  // exact: both are small integers plus the magic
  const T2 r = __hfma2(q, *reinterpret_cast<const T2*>(&s2), *reinterpret_cast<const T2*>(&b2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// 8 consecutive codes of a 4-bit word -> 8 reconstructed 16-bit weights.
template <typename AT>
__device__ __forceinline__ uint4 dequant_word4(uint32_t w, uint32_t s2, uint32_t b2) {
  const uint32_t sh = w >> 4;
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // low half <- byte j of w (code 2j in bits 0..3), high half <- byte j of
    // w >> 4 (code 2j+1 in bits 16..19)
    const uint32_t sel = uint32_t(j) | (uint32_t(j) << 4) | (uint32_t(4 + j) << 8) |
                         (uint32_t(4 + j) << 12);
    const uint32_t t = __byte_perm(w, sh, sel);
    out[j] = fma_pair<AT>((t & 0x000F000Fu) | Act<AT>::kMagic2, s2, b2);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// 4 codes of an 8-bit word -> 2 pairs.
template <typename AT>
__device__ __forceinline__ void dequant_word8(uint32_t w, uint32_t s2, uint32_t b2,
                                              uint32_t& p0, uint32_t& p1);

template <>
__device__ __forceinline__ void dequant_word8<__half>(uint32_t w, uint32_t s2, uint32_t b2,
                                                      uint32_t& p0, uint32_t& p1) {
  // 0x64 in the high byte of each half: 1024 + code, exact for codes < 1024
  p0 = fma_pair<__half>(__byte_perm(w, 0x64646464u, 0x4140u), s2, b2);
  p1 = fma_pair<__half>(__byte_perm(w, 0x64646464u, 0x4342u), s2, b2);
}

template <>
__device__ __forceinline__ void dequant_word8<__nv_bfloat16>(uint32_t w, uint32_t s2, uint32_t b2,
                                                             uint32_t& p0, uint32_t& p1) {
  // bfloat16 has 8 significant bits, too few for 128 + code; go through f32:
  // 2^23 + code is exact, the subtraction is exact, and the code (< 256) is
  // exact in bfloat16.
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | uint32_t(i))) - 8388608.0f;
  const __nv_bfloat162 q01 = __floats2bfloat162_rn(f[0], f[1]);
  const __nv_bfloat162 q23 = __floats2bfloat162_rn(f[2], f[3]);
  const __nv_bfloat162 s = *reinterpret_cast<const __nv_bfloat162*>(&s2);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&b2);
  const __nv_bfloat162 r0 = __hfma2(q01, s, b), r1 = __hfma2(q23, s, b);
  p0 = *reinterpret_cast<const uint32_t*>(&r0);
  p1 = *reinterpret_cast<const uint32_t*>(&r1);
}

// ---- bfloat16 residual operand
// For a pair of weights with codes q (exact, as float), scale s and bias b in
// float32, and hi = RNE_bf16(q*s + b) (the pair as computed above):
//   d  = RNE_f32(q*s + b) - hi          (exact: the two are within 2^-8)
//   lo = RZ_bf16(RNE_f32(d * (1 - 2^-9)))
// Then |hi + lo - (q*s + b)| <= about 2^-15 |q*s + b|, and |lo| stays below
// half a bfloat16 step of hi (the factor keeps it there when the float32
// rounding lands exactly on a midpoint), so hi + lo, accumulated in float32
// and rounded to bfloat16, is hi again: a one-hot x still reproduces the
// reconstruction bit for bit.
__device__ __forceinline__ uint32_t lo_pair(float2 q, float2 s, float2 b, uint32_t hi) {
  const float2 fw = __ffma2_rn(q, s, b);
  const float2 h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
  const float2 d = __ffma2_rn(h, make_float2(-1.0f, -1.0f), fw);
  const float2 dc = __fmul2_rn(d, make_float2(0.998046875f, 0.998046875f));
  uint32_t r;
  // the first source goes to the upper half
  asm("cvt.rz.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(dc.y), "f"(dc.x));
  return r;
}

// 8 codes of a 4-bit word -> hi and lo of 8 bfloat16 weights.
__device__ __forceinline__ void dequant_word4_split(uint32_t w, uint32_t s2, uint32_t b2, float2 sf,
                                                    float2 bf, uint32_t (&hi)[4],
                                                    uint32_t (&lo)[4]) {
  const uint32_t sh = w >> 4;
  const uint32_t mq = Act<__nv_bfloat16>::kMagic2;
  const __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&mq);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t sel = uint32_t(j) | (uint32_t(j) << 4) | (uint32_t(4 + j) << 8) |
                         (uint32_t(4 + j) << 12);
    const uint32_t mp = (__byte_perm(w, sh, sel) & 0x000F000Fu) | Act<__nv_bfloat16>::kMagic2;
    const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&mp), m);
    const __nv_bfloat162 r = __hfma2(q, *reinterpret_cast<const __nv_bfloat162*>(&s2),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b2));
    const uint32_t qb = *reinterpret_cast<const uint32_t*>(&q);
    hi[j] = *reinterpret_cast<const uint32_t*>(&r);
    lo[j] = lo_pair(make_float2(__uint_as_float(qb << 16), __uint_as_float(qb & 0xffff0000u)), sf,
                    bf, hi[j]);
  }
}

// 4 codes of an 8-bit word -> hi and lo of 4 bfloat16 weights (two pairs).
__device__ __forceinline__ void dequant_word8_split(uint32_t w, uint32_t s2, uint32_t b2, float2 sf,
                                                    float2 bf, uint32_t& h0, uint32_t& h1,
                                                    uint32_t& l0, uint32_t& l1) {
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    f[i] = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | uint32_t(i))) - 8388608.0f;
  const __nv_bfloat162 q01 = __floats2bfloat162_rn(f[0], f[1]);
  const __nv_bfloat162 q23 = __floats2bfloat162_rn(f[2], f[3]);
  const __nv_bfloat162 s = *reinterpret_cast<const __nv_bfloat162*>(&s2);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&b2);
  const __nv_bfloat162 r0 = __hfma2(q01, s, b), r1 = __hfma2(q23, s, b);
  h0 = *reinterpret_cast<const uint32_t*>(&r0);
  h1 = *reinterpret_cast<const uint32_t*>(&r1);
  l0 = lo_pair(make_float2(f[0], f[1]), sf, bf, h0);
  l1 = lo_pair(make_float2(f[2], f[3]), sf, bf, h1);
}

// ---- split-K reduction
// Asynchronous 16-byte store into another CTA's shared memory; its bytes are
// counted (complete_tx) on that CTA's mbarrier `bar` (a shared::cluster
// address too).
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float a, float b, float c, float d,
                                               uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(addr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
      : "memory");
}

template <typename AT>
__device__ __forceinline__ uint32_t splat(AT v) {
  const uint16_t u = *reinterpret_cast<const uint16_t*>(&v);
  return uint32_t(u) | (uint32_t(u) << 16);
}

// The 64 reconstructed weights of row r of a stage's packed tile (two per
// register, k ascending) and, for bfloat16, their residuals (lo_pair): the
// reconstruction of qlin_dequant, bit for bit.  Rows past N (row_ok false)
// give zeros.
template <int BITS, typename AT, int kSplit>
__device__ __forceinline__ void dequant_row(const uint8_t* wrow, int r, AT sc, AT bc, bool row_ok,
                                            uint32_t (&a)[32], uint32_t (&lo)[kSplit == 2 ? 32 : 1]) {
  const uint32_t s2 = row_ok ? splat(sc) : 0u, b2 = row_ok ? splat(bc) : 0u;
  if constexpr (kSplit == 2) {
    const float sv = row_ok ? Act<AT>::to_f32(sc) : 0.0f;
    const float bv = row_ok ? Act<AT>::to_f32(bc) : 0.0f;
    const float2 sf = make_float2(sv, sv), bf = make_float2(bv, bv);
    if constexpr (BITS == 4) {
      const int sw = (r >> 2) & 1;
      const uint4 v0 = *reinterpret_cast<const uint4*>(wrow + ((0 ^ sw) << 4));
      const uint4 v1 = *reinterpret_cast<const uint4*>(wrow + ((1 ^ sw) << 4));
      const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c)
        dequant_word4_split(words[c], s2, b2, sf, bf,
                            *reinterpret_cast<uint32_t(*)[4]>(a + 4 * c),
                            *reinterpret_cast<uint32_t(*)[4]>(lo + 4 * c));
    } else {
      const int sw = (r >> 1) & 3;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((c ^ sw) << 4));
        const uint32_t ws4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dequant_word8_split(ws4[e], s2, b2, sf, bf, a[8 * c + 2 * e], a[8 * c + 2 * e + 1],
                              lo[8 * c + 2 * e], lo[8 * c + 2 * e + 1]);
      }
    }
  } else if constexpr (BITS == 4) {
    // packed rows are 32 bytes in the 32-byte TMA swizzle: chunk c of row
    // r sits at chunk c ^ ((r >> 2) & 1)
    const int sw = (r >> 2) & 1;
    const uint4 v0 = *reinterpret_cast<const uint4*>(wrow + ((0 ^ sw) << 4));
    const uint4 v1 = *reinterpret_cast<const uint4*>(wrow + ((1 ^ sw) << 4));
    const uint32_t words[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 o = dequant_word4<AT>(words[c], s2, b2);
      a[4 * c] = o.x;
      a[4 * c + 1] = o.y;
      a[4 * c + 2] = o.z;
      a[4 * c + 3] = o.w;
    }
  } else {
    // packed rows are 64 bytes in the 64-byte TMA swizzle: chunk c of row
    // r sits at chunk c ^ ((r >> 1) & 3)
    const int sw = (r >> 1) & 3;
    uint32_t words[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((c ^ sw) << 4));
      words[4 * c] = v.x;
      words[4 * c + 1] = v.y;
      words[4 * c + 2] = v.z;
      words[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      dequant_word8<AT>(words[2 * c], s2, b2, a[4 * c], a[4 * c + 1]);
      dequant_word8<AT>(words[2 * c + 1], s2, b2, a[4 * c + 2], a[4 * c + 3]);
    }
  }
}

template <int BITS, typename AT, int BN, bool SCALE_TMA>
__global__ void __launch_bounds__(kThreads, 1)
    qmm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_b,
               const AT* __restrict__ scales, const AT* __restrict__ biases, AT* __restrict__ y,
               int M, int N, int K, int stages, int tmem_cols, int split,
               const AT* __restrict__ layer_bias, int y_f32) {
  constexpr int kSplit = OperandSplit<AT>::value;
  using L = Layout<BITS, BN, kSplit, SCALE_TMA>;
  using G = Geo<BITS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb_count = K / kBK;
  const int n_tiles = (N + kBM - 1) / kBM, m_tiles = (M + BN - 1) / BN;
  const int total_tiles = n_tiles * m_tiles;
  // split == 1: persistent CTAs walk tiles blockIdx.x, + gridDim.x, ...
  // split  > 1: a cluster of `split` CTAs shares one tile (grid = tiles x
  // split), CTA `rank` taking k-blocks [kb0, kb1); the partial accumulators
  // are summed through distributed shared memory at the end.
  const int rank = split > 1 ? int(ptx::cluster_ctarank()) : 0;
  const int t_first = int(blockIdx.x) / split, t_step = int(gridDim.x) / split;
  const int kb0 = rank * kb_count / split, kb1 = (rank + 1) * kb_count / split;

  // stage s: [x tile][packed tile][scales][biases]
  auto x_addr = [&](int s) { return base + uint32_t(s * L::kStageBytes); };
  auto w_addr = [&](int s) { return x_addr(s) + uint32_t(L::kWOff); };
  auto s_addr = [&](int s) { return x_addr(s) + uint32_t(L::kSOff); };
  const uint32_t bar_base = base + uint32_t(stages * L::kStageBytes);
  // one "loaded" barrier per stage and dequantising group: use u of the ring
  // (stage u % stages) signals the barrier of group u % kDequantGroups
  auto full_bar = [&](int g, int s) { return bar_base + 8u * (g * stages + s); };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kDequantGroups * stages + s); };
  auto afull_bar = [&](int s) { return bar_base + 8u * ((kDequantGroups + 1) * stages + s); };
  const uint32_t accf_bar = bar_base + 8u * ((kDequantGroups + 2) * stages);  // [2] MMA -> epilogue
  const uint32_t acce_bar = accf_bar + 16u;                   // [2] epilogue -> MMA
  const uint32_t done_bar = acce_bar + 16u;
  const uint32_t red_bar = done_bar + 8u;  // split-K: partials received
  const uint32_t tmem_slot = red_bar + 8u;
  uint32_t* tmem_slot_ptr = reinterpret_cast<uint32_t*>(gbase + (tmem_slot - base));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      for (int g = 0; g < kDequantGroups; ++g) ptx::mbar_init(full_bar(g, s), 1);
      ptx::mbar_init(empty_bar(s), 1 + 4);  // MMA commit + the 4 warps of the dequant group
      ptx::mbar_init(afull_bar(s), 4);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(accf_bar + 8u * b, 1);
      ptx::mbar_init(acce_bar + 8u * b, 4);  // the epilogue warps
    }
    ptx::mbar_init(done_bar, 1);
    ptx::mbar_init(red_bar, 1);
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tm_x);
    ptx::tma_prefetch_desc(&tm_w);
    if constexpr (SCALE_TMA) {
      ptx::tma_prefetch_desc(&tm_s);
      ptx::tma_prefetch_desc(&tm_b);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, uint32_t(tmem_cols));
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;
  // programmatic dependent launch (QLIN_OVERLAP_PREVIOUS): the set-up above
  // ran while the preceding kernel finished; the next kernel may launch now.
  // Both calls are no-ops in a plain launch.
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0, g = 0, issued = 0;
      uint32_t round = 0;
      uint32_t full_ph = 0;  // bit g*8+s: parity of the next phase of full_bar(g, s)
      bool ok = true;
      grid_dependency_wait();  // x is the preceding kernel's output
      for (int t = t_first; t < total_tiles && ok; t += t_step) {
        const int n0 = (t % n_tiles) * kBM, m0 = (t / n_tiles) * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (round > 0 && !ptx::mbar_wait(empty_bar(s), (round - 1) & 1u)) {
            report(kStatusProducer);
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(g, s);
          ptx::mbar_arrive_expect_tx(fb, L::kTxBytes + (SCALE_TMA ? L::kSBytes : 0));
          ptx::tma_load_2d(x_addr(s), &tm_x, fb, kb * kBK, m0);
          ptx::tma_load_2d(w_addr(s), &tm_w, fb, kb * G::kWordsPerGroup, n0);
          if constexpr (SCALE_TMA) {
            // the 8 groups holding group kb (x coordinate a multiple of 8 groups = 16 bytes)
            ptx::tma_load_2d(s_addr(s), &tm_s, fb, kb & ~7, n0);
            ptx::tma_load_2d(s_addr(s) + uint32_t(kBM * 16), &tm_b, fb, kb & ~7, n0);
          }
          full_ph ^= 1u << (g * 8 + s);
          ++issued;
          if (++g == kDequantGroups) g = 0;
          if (++s == stages) {
            s = 0;
            ++round;
          }
        }
      }
      if (!ok) {
        // the last min(issued, stages) loads, one per stage, may be in flight:
        // wait (bounded) for each before the CTA exits
        const int first = issued > stages ? issued - stages : 0;
        for (int v = first; v < issued; ++v) {
          const int vg = v % kDequantGroups, vs = v % stages;
          const uint32_t parity = ((full_ph >> (vg * 8 + vs)) & 1u) ^ 1u;
          if (!ptx::mbar_wait(full_bar(vg, vs), parity)) report(kStatusTeardown);
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = std::is_same<AT, __half>::value ? 0u : 1u;
      constexpr uint32_t idesc = ptx::idesc_f16(fmt, kBM, BN);
      int s = 0, i = 0;
      uint32_t round = 0;
      bool ok = true, any = false;
      for (int t = t_first; t < total_tiles && ok; t += t_step, ++i) {
        const int buf = i % L::kDBufs;
        if (i >= L::kDBufs &&
            !ptx::mbar_wait(acce_bar + 8u * buf, uint32_t(i / L::kDBufs - 1) & 1u)) {
          report(kStatusMma);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(buf * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          // A ready implies the stage's TMA bytes (x included) have landed:
          // the dequantising warps arrive on afull only after they have
          // waited for the stage's full barrier.  One wait per stage: this
          // thread's own latency is part of the stage time.
          if (!ptx::mbar_wait(afull_bar(s), round & 1u)) {
            report(kStatusMma);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_tmem =
              tmem_base + uint32_t(L::kACol0 + s * L::kAColsPerStage);
          const uint64_t bd = ptx::sw128_kmajor_desc(x_addr(s));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K = 16 per MMA: 8 TMEM columns of A; +32 bytes of the x rows =
            // +2 in the descriptor's 16-byte address units
            mma_f16_ts(d_tmem, a_tmem + uint32_t(8 * kk), bd + uint64_t(2 * kk), idesc,
                       (kb > kb0 || kk > 0) ? 1u : 0u);
            if constexpr (kSplit == 2)  // the bfloat16 residual lo, 32 columns on
              mma_f16_ts(d_tmem, a_tmem + uint32_t(32 + 8 * kk), bd + uint64_t(2 * kk), idesc, 1u);
          }
          any = true;
          ptx::mma_commit(empty_bar(s));
          if (++s == stages) {
            s = 0;
            ++round;
          }
        }
        if (ok) ptx::mma_commit(accf_bar + 8u * buf);
      }
      // before TMEM is freed every MMA issued here must have completed
      ptx::mma_commit(done_bar);
      if (any && !ptx::mbar_wait(done_bar, 0)) report(kStatusTeardown);
    }
  } else if (warp < 2 + kDequantWarps) {
    // -------------------------------- dequantise (warpgroups take uses in turn)
    // Group g takes the ring uses u with u % kDequantGroups == g and waits on
    // its own barriers full_bar(g, .), whose phases it alone consumes, in
    // order: it can never wait on a phase two ahead of a barrier's last
    // completed one (a parity wait cannot tell those apart), whatever the ring
    // depth.
    const int grp = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row within the tile
    const int gpr = K / kGroup;
    // this thread's TMEM lane (its weight row) at the first A slot
    const uint32_t a_lane = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(L::kACol0);
    int s = 0, u = 0;
    uint32_t full_ph = 0;  // bit s: parity of the next phase of full_bar(grp, s)
    bool ok = true;
    for (int t = t_first; t < total_tiles && ok; t += t_step) {
      const int n = (t % n_tiles) * kBM + r;
      const bool row_ok = n < N;
      const AT* srow = scales + int64_t(min(n, N - 1)) * gpr;
      const AT* brow = biases + int64_t(min(n, N - 1)) * gpr;
      for (int kb = kb0; kb < kb1; ++kb, ++u) {
        const int cs = s;
        if (++s == stages) s = 0;
        if (u % kDequantGroups != grp) continue;
        AT sc, bc;
        if constexpr (!SCALE_TMA) {
          sc = srow[kb];
          bc = brow[kb];
        }
        // warp-uniform outcome: tcgen05.st below needs the whole warp
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(full_bar(grp, cs), (full_ph >> cs) & 1u))) {
          report(kStatusDequant);
          ok = false;
          break;
        }
        full_ph ^= 1u << cs;
        if constexpr (SCALE_TMA) {
          const AT* ss = reinterpret_cast<const AT*>(gbase + (s_addr(cs) - base));
          sc = ss[r * 8 + (kb & 7)];
          bc = ss[kBM * 8 + r * 8 + (kb & 7)];
        }
        const uint8_t* wrow = gbase + (w_addr(cs) - base) + r * G::kPackedRowBytes;
        // the row's 64 reconstructed weights, two per register, k ascending
        // (and, for bfloat16, their residuals)
        uint32_t a[32];
        uint32_t lo[kSplit == 2 ? 32 : 1];
        dequant_row<BITS, AT, kSplit>(wrow, r, sc, bc, row_ok, a, lo);
        // into the stage's A slot; complete before the MMA issuer is told
        tmem_st_32x32b_x32(a_lane + uint32_t(cs * L::kAColsPerStage), a);
        if constexpr (kSplit == 2)
          tmem_st_32x32b_x32(a_lane + uint32_t(cs * L::kAColsPerStage + 32), lo);
        tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(afull_bar(cs));
          ptx::mbar_arrive(empty_bar(cs));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;
    int i = 0;
    grid_dependency_wait();  // y is written only after the preceding kernel
    for (int t = t_first; t < total_tiles; t += t_step, ++i) {
      const int buf = i % L::kDBufs;
      if (!__all_sync(0xffffffffu,
                      ptx::mbar_wait(accf_bar + 8u * buf, uint32_t(i / L::kDBufs) & 1u))) {
        report(kStatusEpilogue);
        break;
      }
      ptx::tc_fence_after();
      if (split > 1) break;  // partial accumulator: reduced across the cluster below
      const int n = (t % n_tiles) * kBM + r, m0 = (t / n_tiles) * BN;
      // a linear layer's bias (qlin_linear_ex) joins the f32 sum before the rounding
      const float lb = layer_bias && n < N ? Act<AT>::to_f32(layer_bias[n]) : 0.0f;
      const uint32_t t_lane = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(buf * BN);
      // batches of up to 64 columns: four loads, one wait (a TMEM load's
      // latency per batch, not per 16 columns); the accumulator is handed
      // back to the MMA issuer as soon as the last batch is in registers
      constexpr int kBatch = BN < 64 ? BN : 64;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += kBatch) {
        uint32_t v[kBatch];
#pragma unroll
        for (int c = 0; c < kBatch; c += 16)
          ptx::tmem_ld_32x32b_x16(t_lane + uint32_t(c0 + c),
                                  *reinterpret_cast<uint32_t(*)[16]>(v + c));
        ptx::tmem_wait_ld();
        if (c0 + kBatch >= BN) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(acce_bar + 8u * buf);
        }
        if (n < N) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int m = m0 + c0 + j;
            const float o = __uint_as_float(v[j]) + lb;
            if (m < M) {
              if (y_f32)
                reinterpret_cast<float*>(y)[int64_t(m) * N + n] = o;
              else
                y[int64_t(m) * N + n] = Act<AT>::from_f32_rn(o);
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();

  if (split > 1) {
    // ---------------------------------------------- split-K reduction
    // The tile's BN columns are cut into `split` slices; CTA d owns slice d.
    // Every CTA sends its partial of each other slice d to CTA d's shared
    // memory (the ring, idle once every CTA of the cluster is past its K
    // loop): receive buffer [split-1 sources][slice/4][128 rows] of float4,
    // row-minor so that a warp's 16-byte stores fall in distinct banks.
    // Each owner then adds the partials in a fixed order (its own first,
    // then the sources by rank) and stores its slice.
    // Eight warps share the work: the four epilogue warps and the first
    // dequantising warpgroup (idle by now), one of each per TMEM lane quarter.
    // Part p of a quarter takes columns [p * half, p * half + half) of every
    // slice (one part when a slice has fewer than 32 columns).
    const int slice = BN / split;
    const int parts = slice >= 32 ? 2 : 1;
    const int half = slice / parts;
    const bool tile = t_first < total_tiles;
    const bool epi_warp = warp >= 2 + kDequantWarps;
    const bool helper_warp = warp >= 2 && warp < 2 + 4;  // dequant warpgroup 0
    const int part = epi_warp ? 0 : 1;
    const bool red = tile && (epi_warp || (helper_warp && parts == 2));
    const int col0 = part * half;
    // arm the receive barrier with every byte the other CTAs will send
    // before any of them can start (the cluster barrier below)
    if (threadIdx.x == 0 && tile)
      ptx::mbar_arrive_expect_tx(red_bar, uint32_t((split - 1) * slice * kBM * 4));
    ptx::cluster_sync();  // every CTA of the cluster is past its K loop and armed
    // (the accumulator is complete: the epilogue warps saw its commit before
    // the CTA barrier; TMEM loads follow the thread synchronisation)
    ptx::tc_fence_after();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + (uint32_t(quarter * 32) << 16);
    // batches of up to 64 columns: four TMEM loads, one wait
    constexpr int kRBatch = BN < 64 ? BN : 64;
    const int batch = half < kRBatch ? half : kRBatch;
    if (red) {
      for (int d = 0; d < split; ++d) {
        if (d == rank) continue;
        const int slot = rank < d ? rank : rank - 1;
        const uint32_t dst =
            ptx::map_shared_rank(base, uint32_t(d)) + uint32_t(slot * (slice / 4) * kBM * 16);
        const uint32_t dst_bar = ptx::map_shared_rank(red_bar, uint32_t(d));
#pragma unroll 1
        for (int c0 = col0; c0 < col0 + half; c0 += batch) {
          uint32_t v[kRBatch];
#pragma unroll
          for (int c = 0; c < kRBatch; c += 16)
            if (c < batch)
              ptx::tmem_ld_32x32b_x16(t_lane + uint32_t(d * slice + c0 + c),
                                      *reinterpret_cast<uint32_t(*)[16]>(v + c));
          ptx::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < kRBatch / 4; ++q)
            if (q < batch / 4)
              st_async_f32x4(dst + uint32_t(((c0 / 4 + q) * kBM + r) * 16),
                             __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                             __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]),
                             dst_bar);
        }
      }
    }
    // every partial destined to this CTA has landed (bounded wait)
    const bool got = !red || __all_sync(0xffffffffu, ptx::mbar_wait(red_bar, 0));
    if (!got) report(kStatusEpilogue);
    // (the block runs whether or not the wait succeeded: its named barrier
    // needs all the reducing warps; a timeout is reported, the values are
    // then garbage)
    if (red) {
      // sum into f16/bf16, stage [slice tokens][128 rows] in shared memory
      // (after the receive buffer), then store y with 16-byte vectors
      const int t = t_first;
      const int n0 = (t % n_tiles) * kBM, m0 = (t / n_tiles) * BN + rank * slice;
      AT* stage_y = reinterpret_cast<AT*>(gbase + (split - 1) * slice * kBM * 4);
      const float lb = layer_bias && n0 + r < N ? Act<AT>::to_f32(layer_bias[n0 + r]) : 0.0f;
#pragma unroll 1
      for (int c0 = col0; c0 < col0 + half; c0 += batch) {
        uint32_t v[kRBatch];
#pragma unroll
        for (int c = 0; c < kRBatch; c += 16)
          if (c < batch)
            ptx::tmem_ld_32x32b_x16(t_lane + uint32_t(rank * slice + c0 + c),
                                    *reinterpret_cast<uint32_t(*)[16]>(v + c));
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kRBatch / 4; ++q) {
          if (q < batch / 4) {
            float a0 = __uint_as_float(v[4 * q]), a1 = __uint_as_float(v[4 * q + 1]);
            float a2 = __uint_as_float(v[4 * q + 2]), a3 = __uint_as_float(v[4 * q + 3]);
            for (int src = 0; src < split - 1; ++src) {
              const float4 p = *reinterpret_cast<const float4*>(
                  gbase + ((src * (slice / 4) + c0 / 4 + q) * kBM + r) * 16);
              a0 += p.x;
              a1 += p.y;
              a2 += p.z;
              a3 += p.w;
            }
            const int mm = c0 + 4 * q;
            a0 += lb;
            a1 += lb;
            a2 += lb;
            a3 += lb;
            if (y_f32) {
              // float32 output: stored directly, rows along n
              float* yf = reinterpret_cast<float*>(y);
              const int n = n0 + r;
              if (n < N) {
                if (m0 + mm < M) yf[int64_t(m0 + mm) * N + n] = a0;
                if (m0 + mm + 1 < M) yf[int64_t(m0 + mm + 1) * N + n] = a1;
                if (m0 + mm + 2 < M) yf[int64_t(m0 + mm + 2) * N + n] = a2;
                if (m0 + mm + 3 < M) yf[int64_t(m0 + mm + 3) * N + n] = a3;
              }
              continue;
            }
            stage_y[(mm + 0) * kBM + r] = Act<AT>::from_f32_rn(a0);
            stage_y[(mm + 1) * kBM + r] = Act<AT>::from_f32_rn(a1);
            stage_y[(mm + 2) * kBM + r] = Act<AT>::from_f32_rn(a2);
            stage_y[(mm + 3) * kBM + r] = Act<AT>::from_f32_rn(a3);
          }
        }
      }
      // every reducing warp's columns are staged (the same branch for all of
      // them: y_f32 is a kernel argument)
      if (!y_f32) {
        const int n_red = 128 * parts;  // threads of the reducing warps
        if (parts == 2)
          asm volatile("bar.sync 2, 256;" ::: "memory");
        else
          asm volatile("bar.sync 2, 128;" ::: "memory");
        const int et = part * 128 + quarter * 32 + lane;  // 0 .. n_red-1
        const bool vec = N % 8 == 0 && n0 + kBM <= N &&
                         reinterpret_cast<uintptr_t>(y) % 16 == 0;
        if (vec) {
          // 16 chunks of 8 rows per token
#pragma unroll 1
          for (int c = et; c < slice * 16; c += n_red) {
            const int mm = c >> 4, n8 = (c & 15) * 8;
            if (m0 + mm < M)
              *reinterpret_cast<uint4*>(y + int64_t(m0 + mm) * N + n0 + n8) =
                  *reinterpret_cast<const uint4*>(stage_y + mm * kBM + n8);
          }
        } else {
          const int n = n0 + r;
          if (n < N)
            for (int mm = col0; mm < col0 + half; ++mm)
              if (m0 + mm < M) y[int64_t(m0 + mm) * N + n] = stage_y[mm * kBM + r];
        }
      }
    }
    // no CTA leaves while another may still be writing into it
    ptx::cluster_sync();
    ptx::tc_fence_before();
    __syncthreads();
  }

  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, uint32_t(tmem_cols));
  }
}

// ------------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

qlin_status make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(QLIN_ERR_CUDA, "qlin_qmm: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(QLIN_ERR_CUDA, "qlin_qmm: cuTensorMapEncodeTiled failed (%d)", int(r));
  return QLIN_OK;
}

template <int BITS, typename AT, int BN, bool SCALE_TMA>
qlin_status launch_layout(const void* x, const uint32_t* wq, const void* scales,
                          const void* biases, void* y, int64_t M, int64_t N, int64_t K, int split,
                          const Epilogue& ep, unsigned flags, cudaStream_t st) {
  using L = Layout<BITS, BN, OperandSplit<AT>::value, SCALE_TMA>;
  constexpr int kMaxSmem = 227 * 1024;
  constexpr int kBarBytes = 512;
  // (kDequantGroups + 2) barriers per stage (at most 8), two pairs of
  // accumulator barriers, the teardown barrier and the TMEM address slot
  static_assert((kDequantGroups + 2) * 8 * 8 + 4 * 8 + 8 + 8 + 4 <= kBarBytes, "barrier block");
  int stages =
      std::min(std::min(8, L::kMaxStages), (kMaxSmem - 1024 - kBarBytes) / L::kStageBytes);
  // QLIN_QMM_STAGES (2..8) caps the ring depth, for tuning
  if (const char* env = std::getenv("QLIN_QMM_STAGES")) {
    const int v = std::atoi(env);
    if (v >= 2 && v < stages) stages = v;
  }
  if (stages < 2) return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmm: tile does not fit");
  // split-K: slices of at least 16 columns, and the receive buffer of the
  // reduction fits in the ring
  if (split > 1 && (BN / split < 16 || BN % split != 0 ||
                    (split - 1) * kBM * (BN / split) * 4 + (BN / split) * kBM * 2 >
                        stages * L::kStageBytes))
    split = 1;
  const size_t smem = size_t(stages) * L::kStageBytes + 1024 + kBarBytes;
  // TMEM columns: the accumulators and one A slot per stage, rounded up to a
  // power of two (tcgen05.alloc); at most 512
  int tmem_cols = 32;
  while (tmem_cols < L::kACol0 + stages * L::kAColsPerStage) tmem_cols *= 2;
  if (tmem_cols > 512) return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmm: TMEM layout does not fit");

  CUtensorMap tm_x, tm_w, tm_s, tm_b;
  const CUtensorMapDataType adt = std::is_same<AT, __half>::value
                                      ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  qlin_status s = make_map(&tm_x, adt, x, uint64_t(K), uint64_t(M), uint64_t(K) * 2, kBK, BN,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  if (s != QLIN_OK) return s;
  const uint64_t wpr = uint64_t(K) * BITS / 32;
  s = make_map(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, wpr, uint64_t(N), wpr * 4,
               Geo<BITS>::kWordsPerGroup, kBM,
               BITS == 4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (s != QLIN_OK) return s;
  if constexpr (SCALE_TMA) {
    const uint64_t gpr = uint64_t(K) / kGroup;
    if ((s = make_map(&tm_s, adt, scales, gpr, uint64_t(N), gpr * 2, 8, kBM,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) != QLIN_OK)
      return s;
    if ((s = make_map(&tm_b, adt, biases, gpr, uint64_t(N), gpr * 2, 8, kBM,
                      CU_TENSOR_MAP_SWIZZLE_NONE)) != QLIN_OK)
      return s;
  } else {
    tm_s = tm_x;  // unused
    tm_b = tm_x;
  }

  auto kern = qmm_kernel<BITS, AT, BN, SCALE_TMA>;
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
        cudaSuccess)
      return check_launch("qlin_qmm: cudaFuncSetAttribute");
    attr_dev = dev;
  }
  const int64_t tiles = ((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  if (tiles > (int64_t(1) << 30)) return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmm: too many tiles");
  // persistent (one CTA per SM) or, split-K, one cluster of `split` CTAs per tile
  const int64_t grid = split > 1 ? tiles * split : std::min<int64_t>(tiles, sm_count());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1u, 1u);
  cfg.blockDim = dim3(unsigned(kThreads), 1u, 1u);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  if (split > 1) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = unsigned(split);
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (flags & QLIN_OVERLAP_PREVIOUS) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, kern, tm_x, tm_w, tm_s, tm_b, static_cast<const AT*>(scales),
      static_cast<const AT*>(biases), static_cast<AT*>(y), int(M), int(N), int(K), stages,
      tmem_cols, split, static_cast<const AT*>(ep.bias), ep.y_f32);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QLIN_ERR_CUDA, "qmm_kernel launch: %s", cudaGetErrorString(e));
  }
  return check_launch("qmm_kernel");
}

// Scales and biases by TMA boxes of 8 groups x 128 rows (needs 16-byte
// rows), of which a stage uses one group, for rows of more than 32 groups.
// For rows of at most 32 groups (K <= 2048) the dequantising threads read
// their row's scale and bias from global memory instead (L1 holds the row's
// 64 bytes of each for all its stages; the loads are issued before the
// stage's barrier wait), and the stages, 4 KB smaller without the boxes, make
// room for a sixth at 4 bits: 2-6% faster there (8192 x 2048 at M = 2048:
// 62.8 -> 61.1 us at 4 bits, 62.3 -> 58.8 at 8 bits), while at K = 8192 the
// boxes are 3-9% faster.
template <int BITS, typename AT, int BN>
qlin_status launch_bn(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                      void* y, int64_t M, int64_t N, int64_t K, int split, const Epilogue& ep,
                      unsigned flags, cudaStream_t st) {
  const uint64_t gpr = uint64_t(K) / kGroup;
  const bool scale_tma = gpr > 32 && gpr % 8 == 0 &&
                         reinterpret_cast<uintptr_t>(scales) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(biases) % 16 == 0;
  return scale_tma ? launch_layout<BITS, AT, BN, true>(x, wq, scales, biases, y, M, N, K, split,
                                                       ep, flags, st)
                   : launch_layout<BITS, AT, BN, false>(x, wq, scales, biases, y, M, N, K,
                                                        split, ep, flags, st);
}

template <int BITS, typename AT>
qlin_status dispatch(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, const Epilogue& ep,
                     unsigned flags, cudaStream_t st) {
  // Token tile and split-K factor: the pair with the smallest estimated time,
  // waves of tiles x stages per CTA x time per stage, + the reduction when K
  // is split.  Measured on GB300 for every tile from 32 to 256 tokens, a
  // 64-k stage takes about 0.43 us whatever BN (the MMAs of a 256-token stage
  // alone take 0.26 us; the stage's trip through the ring sets the rate).  So
  // wider tiles are free and narrower ones only pay when they remove a wave.  K is split over a
  // cluster of 2 or 4 CTAs only when the split tiles fit on the SMs at once
  // and leave each CTA at least 4 stages; the reduction costs about 2.5 us +
  // 0.045 us per accumulator column a CTA sends.  Ties go to the larger tile.
  // Tiles wider than the batch are candidates too: the rows past M are
  // zero-filled by the TMA without memory traffic, cost the MMA nothing, and
  // a wider tile can be split over more CTAs.
  const int max_bn = 256;
  const int64_t sms = sm_count();
  const int64_t n_tiles = (N + kBM - 1) / kBM;
  const int64_t kb_count = K / kBK;
  int bn = max_bn, split = 1;
  double best = -1.0;
  for (int cand = max_bn; cand >= 16; cand >>= 1) {
    const int64_t tiles = n_tiles * ((M + cand - 1) / cand);
    // (bfloat16 issues twice the MMAs per stage: the residual operand)
    const double t_stage = OperandSplit<AT>::value == 2 ? 0.75 : 0.43;
    for (int sp = 1; sp <= 4; sp *= 2) {
      if (sp > 1 && (tiles * sp > sms || kb_count < 4 * sp || cand / sp < 16)) continue;
      const int64_t waves = (tiles * sp + sms - 1) / sms;
      // the reduction: about 2.5 us + 0.045 us per column each CTA sends
      const double cost = double(waves) * double((kb_count + sp - 1) / sp) * t_stage +
                          (sp > 1 ? 2.5 + 0.045 * cand * (sp - 1) / sp : 0.0);
      if (best < 0.0 || cost < best * 0.97) {
        best = cost;
        bn = cand;
        split = sp;
      }
    }
  }
  // QLIN_QMM_BN (16, 32, 64, 128 or 256) and QLIN_QMM_SPLIT (1, 2 or 4)
  // override the choice, for tuning
  if (const char* env = std::getenv("QLIN_QMM_BN")) {
    const int v = std::atoi(env);
    if (v == 16 || v == 32 || v == 64 || v == 128 || v == 256) bn = v;
  }
  if (const char* env = std::getenv("QLIN_QMM_SPLIT")) {
    const int v = std::atoi(env);
    if (v == 1 || v == 2 || v == 4) split = v;
  }
  switch (bn) {
    case 16: return launch_bn<BITS, AT, 16>(x, wq, scales, biases, y, M, N, K, split, ep, flags,
                                               st);
    case 32: return launch_bn<BITS, AT, 32>(x, wq, scales, biases, y, M, N, K, split, ep, flags,
                                               st);
    case 64: return launch_bn<BITS, AT, 64>(x, wq, scales, biases, y, M, N, K, split, ep, flags,
                                               st);
    case 128: return launch_bn<BITS, AT, 128>(x, wq, scales, biases, y, M, N, K, split, ep, flags,
                                               st);
    default: return launch_bn<BITS, AT, 256>(x, wq, scales, biases, y, M, N, K, split, ep, flags,
                                              st);
  }
}

}  // namespace

qlin_status launch_qmm(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       unsigned flags, const Epilogue& ep, cudaStream_t st) {
  if (dtype == QLIN_F16)
    return bits == 4 ? dispatch<4, __half>(x, wq, scales, biases, y, M, N, K, ep, flags, st)
                     : dispatch<8, __half>(x, wq, scales, biases, y, M, N, K, ep, flags, st);
  return bits == 4
             ? dispatch<4, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, ep, flags, st)
             : dispatch<8, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, ep, flags, st);
}

cudaError_t qmm_take_device_status(unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qmm_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_qmm_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace qlin
