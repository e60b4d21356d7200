// Device building blocks shared by the CUDA-core qmv kernels (single launch
// and decode-step chain).
//
// Arithmetic (f32 throughout, one RNE to the output type at the end):
//   A 16-byte chunk of a row holds CW = 128/bits codes sharing one group
//   (64 % CW == 0).  Each code becomes the float MAGIC + q by placing it under
//   the exponent of MAGIC (4-bit: 128.0f, code bits 16..19; 8-bit: 32768.0f,
//   code bits 8..15): one byte permute per code, exact.  Per chunk, with
//   f32x2 FMAs over (even, odd) code positions,
//       P = sum_k x_k * (MAGIC + q_k),   X = sum_k x_k
//       sum_k x_k * w_hat_k = scale * (P - MAGIC * X) + bias * X
//   (w_hat = q*scale + bias: "track(upstream-iree): fused dequant->matmul for
//   the packed int8 bandwidth win", section "What is already in-tree").  X
//   (split even/odd) is computed once per CTA and shared by all rows.  The
//   cancellation in P - MAGIC*X costs log2(MAGIC / mean code) bits of the 24
//   (about 4 for 4-bit, 8 for 8-bit), far inside the output tolerance.
//
// x lives in shared memory as f32 in a lane-transposed layout
// ([round][4-code group][lane][4]) so that lanes reading consecutive 16-byte
// chunks of a row read consecutive 16-byte words of x: conflict-free.
#pragma once

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace qmvcore {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;

template <int BITS>
struct Unpack;

// 4-bit: nibbles are spread to bytes (even codes, odd codes), then each byte
// lands in bits 16..19 under the exponent of 128.0f with one byte permute.
template <>
struct Unpack<4> {
  static constexpr int kCodes = 8;  // per word
  static constexpr float kMagic = 128.0f;
  static __device__ __forceinline__ void run(uint32_t w, float2 (&f)[4]) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // codes 0,2,4,6 in bytes 0..3
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes 1,3,5,7
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t sel = 0x7054u | (uint32_t(i) << 8);  // [0, 0, byte i, 0x43]
      f[i].x = u32_as_f32(__byte_perm(lo, 0x43000000u, sel));
      f[i].y = u32_as_f32(__byte_perm(hi, 0x43000000u, sel));
    }
  }
};

// 8-bit: each code byte lands in bits 8..15 under the exponent of 32768.0f
// (0x47000000), whose unit bit is bit 8.
template <>
struct Unpack<8> {
  static constexpr int kCodes = 4;
  static constexpr float kMagic = 32768.0f;
  static __device__ __forceinline__ void run(uint32_t w, float2 (&f)[2]) {
    f[0].x = u32_as_f32(__byte_perm(w, 0x47000000u, 0x7404u));  // [0, byte 0, 0, 0x47]
    f[0].y = u32_as_f32(__byte_perm(w, 0x47000000u, 0x7414u));
    f[1].x = u32_as_f32(__byte_perm(w, 0x47000000u, 0x7424u));
    f[1].y = u32_as_f32(__byte_perm(w, 0x47000000u, 0x7434u));
  }
};

// Halving butterfly: on entry every lane holds V partial values; on exit lane
// l holds the warp-wide sum of value index l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float butterfly_sum(float (&v)[V], int lane) {
  static_assert((V & (V - 1)) == 0 && V <= 32, "V must be a power of two <= 32");
  int off = 16;
#pragma unroll
  for (int nv = V; nv > 1; nv >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int t = 0; t < nv / 2; ++t) {
      const float keep = upper ? v[t + nv / 2] : v[t];
      const float send = upper ? v[t] : v[t + nv / 2];
      v[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// floats of one row of x in the transposed layout
__host__ __device__ constexpr int xs_floats(int rounds, int bits) { return rounds * 32 * (128 / bits); }

// Stage MT rows of x (row stride ldx, rows >= m_valid read as 0) and their
// per-chunk (even, odd) sums.  All consumer threads call it.  L2_ONLY reads x
// through L2 (for data another CTA of the same grid just wrote).  Every thread
// issues all of its 16-byte loads before converting (one memory latency, not
// one per round), and the threads of a chunk (CW/8 consecutive threads) sum
// it with shuffles, so there is a single barrier.
template <int BITS, int MT, typename AT, bool L2_ONLY>
__device__ __forceinline__ void stage_x(const AT* x, int64_t ldx, int m_valid, int K, int rounds,
                                        float* xs, float2* xsum, int tid) {
  constexpr int kCW = 128 / BITS;
  constexpr int kTPC = kCW / 8;      // threads per chunk (2 or 4)
  constexpr int kMaxIter = 4;        // unrolled loads per thread: K <= 8192 at MT = 1
  const int C = K / kCW;
  const int xs_m = xs_floats(rounds, BITS);
  const int total = MT * (K / 8);    // 16-byte pieces of x
  // zero the chunk sums of the padding chunks of the last round
  for (int e = tid; e < MT * rounds * 32; e += kConsumerThreads)
    if (e % (rounds * 32) >= C) xsum[e] = make_float2(0.0f, 0.0f);
  for (int e0 = 0; e0 < total; e0 += kMaxIter * kConsumerThreads) {
    uint4 raw[kMaxIter];
#pragma unroll
    for (int it = 0; it < kMaxIter; ++it) {
      const int e = e0 + it * kConsumerThreads + tid;
      raw[it] = make_uint4(0u, 0u, 0u, 0u);
      if (e < total) {
        const int mm = e / (K / 8), k0 = (e % (K / 8)) * 8;
        if (mm < m_valid) {
          const uint4* src = reinterpret_cast<const uint4*>(x + int64_t(mm) * ldx + k0);
          raw[it] = L2_ONLY ? __ldcg(src) : *src;
        }
      }
    }
#pragma unroll
    for (int it = 0; it < kMaxIter; ++it) {
      const int e = e0 + it * kConsumerThreads + tid;
      // the kTPC threads of a chunk are consecutive lanes of one warp, and
      // e < total is uniform across them (total is a multiple of kTPC)
      const AT* h = reinterpret_cast<const AT*>(&raw[it]);
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = Act<AT>::to_f32(h[j]);
      float2 part = make_float2(v[0] + v[2] + v[4] + v[6], v[1] + v[3] + v[5] + v[7]);
#pragma unroll
      for (int o = 1; o < kTPC; o <<= 1) {
        part.x += __shfl_xor_sync(0xffffffffu, part.x, o);
        part.y += __shfl_xor_sync(0xffffffffu, part.y, o);
      }
      if (e < total) {
        const int mm = e / (K / 8), k0 = (e % (K / 8)) * 8;
        const int c = k0 / kCW, j4 = (k0 % kCW) / 4;
        float* base = xs + mm * xs_m + ((c >> 5) * (kCW / 4) * 32 + (c & 31)) * 4;
        *reinterpret_cast<float4*>(base + j4 * 128) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(base + (j4 + 1) * 128) = make_float4(v[4], v[5], v[6], v[7]);
        if ((tid % kTPC) == 0) xsum[mm * rounds * 32 + c] = part;
      }
    }
  }
  consumers_sync();
}

// One pipeline stage holds RB rows x kt_bytes of packed codes (row r at
// r * kt_bytes), then, when scales/biases were copied, RB x kt_groups scales
// and RB x kt_groups biases.
struct StageGeom {
  int kt_bytes;   // bytes of a row in this k-tile
  int kt_groups;  // groups of a row in this k-tile
  int rounds;     // rounds of the x layout (ceil(chunks per row / 32))
  int gpr;        // groups per row (for scales read from global memory)
  int N;          // rows of the matrix (rows >= N are never stored)
};

// Accumulate one stage into acc for the R rows (block rows w0 .. w0+R-1, global
// rows row0 ..) this warp owns; k-tile kt of the row, which is k-tile kt_x of
// the staged x (kt_x = kt unless x was staged from a later k-tile on).
template <int BITS, int MT, int R, typename AT>
__device__ __forceinline__ void accumulate_stage(const uint8_t* stage, int RB, int w0, int kt,
                                                 int kt_x, const StageGeom& g, bool scale_copy,
                                                 const AT* __restrict__ scales,
                                                 const AT* __restrict__ biases, int row0,
                                                 const float* xs, const float2* xsum, int lane,
                                                 float2 (&acc)[R][MT]) {
  using U = Unpack<BITS>;
  constexpr int kCW = 128 / BITS;
  constexpr int kCPW = U::kCodes;
  const int kt_chunks = g.kt_bytes / 16;
  const int xs_m = xs_floats(g.rounds, BITS);
  const float2 neg_magic = make_float2(-U::kMagic, -U::kMagic);
  const uint8_t* wst = stage + size_t(w0) * g.kt_bytes;
  const AT* sst = reinterpret_cast<const AT*>(stage + size_t(RB) * g.kt_bytes);
  const AT* bst = sst + RB * g.kt_groups;
  for (int cl = lane; cl < kt_chunks; cl += 32) {
    const int c = kt * kt_chunks + cl;   // chunk index within the row
    const int cx = kt_x * kt_chunks + cl;  // chunk index within the staged x
    const int gl = (cl * kCW) / kGroup;  // group within the k-tile
    uint4 cw[R];
    float2 s2[R], b2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      // rows past N were not copied: their values are never stored
      cw[r] = *reinterpret_cast<const uint4*>(wst + size_t(r) * g.kt_bytes + cl * 16);
      float sv, bv;
      if (scale_copy) {
        sv = Act<AT>::to_f32(sst[(w0 + r) * g.kt_groups + gl]);
        bv = Act<AT>::to_f32(bst[(w0 + r) * g.kt_groups + gl]);
      } else {
        const int64_t gi = int64_t(min(row0 + r, g.N - 1)) * g.gpr + (c * kCW) / kGroup;
        sv = Act<AT>::to_f32(scales[gi]);
        bv = Act<AT>::to_f32(biases[gi]);
      }
      s2[r] = make_float2(sv, sv);
      b2[r] = make_float2(bv, bv);
    }
    const float* xbase = xs + ((cx >> 5) * (kCW / 4) * 32 + (cx & 31)) * 4;
    float2 P[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) P[r][mm] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      float2 xv[MT][kCPW / 2];
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int j = 0; j < kCPW / 4; ++j) {
          const float4 t =
              *reinterpret_cast<const float4*>(xbase + mm * xs_m + (wi * (kCPW / 4) + j) * 128);
          xv[mm][2 * j] = make_float2(t.x, t.y);
          xv[mm][2 * j + 1] = make_float2(t.z, t.w);
        }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t word = wi == 0 ? cw[r].x : wi == 1 ? cw[r].y : wi == 2 ? cw[r].z : cw[r].w;
        float2 f[kCPW / 2];
        U::run(word, f);
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
          for (int j = 0; j < kCPW / 2; ++j) P[r][mm] = __ffma2_rn(f[j], xv[mm][j], P[r][mm]);
      }
    }
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) {
      const float2 X = xsum[mm * g.rounds * 32 + cx];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 D = __ffma2_rn(neg_magic, X, P[r][mm]);
        acc[r][mm] = __ffma2_rn(s2[r], D, acc[r][mm]);
        acc[r][mm] = __ffma2_rn(b2[r], X, acc[r][mm]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fast path: k-tiles of exactly 2048 codes per row (K % 2048 == 0) with the
// scales and biases copied into the stage.  Everything the lane loop indexes
// is a compile-time offset from a per-lane base, and each warp converts its
// rows' 32 scales/biases per tile to f32 pairs once, so the per-chunk work is
// the unpack, the FMAs and three 128-bit / one 64-bit shared loads.
template <int BITS>
struct FixedTile {
  static constexpr int kCodes = 2048;               // codes per row per k-tile
  static constexpr int kBytes = kCodes * BITS / 8;  // 1024 (4-bit) or 2048 (8-bit)
  static constexpr int kChunks = kBytes / 16;
  static constexpr int kRounds = kChunks / 32;      // chunks per lane per row
  static constexpr int kGroups = kCodes / kGroup;   // 32
};

// Warp-private f32 (scale, bias) pairs of the warp's R rows for one stage.
template <int BITS, int R, typename AT>
__device__ __forceinline__ void stage_scales_f32(const uint8_t* stage, int RB, int w0,
                                                 float2* sb32, int lane) {
  using T = FixedTile<BITS>;
  const AT* sst = reinterpret_cast<const AT*>(stage + size_t(RB) * T::kBytes);
  const AT* bst = sst + RB * T::kGroups;
  __syncwarp();  // every lane is done with the previous stage's pairs
#pragma unroll
  for (int r = 0; r < R; ++r)
    sb32[r * 32 + lane] = make_float2(Act<AT>::to_f32(sst[(w0 + r) * T::kGroups + lane]),
                                      Act<AT>::to_f32(bst[(w0 + r) * T::kGroups + lane]));
  __syncwarp();
}

// kt: the k-tile of the staged x (the packed tile is the stage itself).
// Rounds [I0, I0 + NI) of the tile (every round by default): a round is the
// 32 consecutive chunks of a row that the warp's lanes take at once.
template <int BITS, int MT, int R, typename AT, int I0 = 0, int NI = FixedTile<BITS>::kRounds>
__device__ __forceinline__ void accumulate_fixed(const uint8_t* stage, int w0, int kt,
                                                 const float2* sb32, const float* xs, int xs_m,
                                                 const float2* xsum, int xsum_m, int lane,
                                                 float2 (&acc)[R][MT]) {
  using U = Unpack<BITS>;
  using T = FixedTile<BITS>;
  constexpr int kCW = 128 / BITS;
  constexpr int kCPW = U::kCodes;
  const float2 neg_magic = make_float2(-U::kMagic, -U::kMagic);
  const uint8_t* wl = stage + size_t(w0) * T::kBytes + lane * 16;
  const float* xl = xs + lane * 4 + kt * T::kRounds * (kCW / 4) * 128;
  const float2* xsl = xsum + kt * T::kChunks + lane;
  const float2* sbl = sb32 + (lane * kCW) / kGroup;
#pragma unroll
  for (int i = I0; i < I0 + NI; ++i) {
    uint4 cw[R];
    float2 s2[R], b2[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      cw[r] = *reinterpret_cast<const uint4*>(wl + r * T::kBytes + i * 512);
      const float2 sb = sbl[r * 32 + i * (32 * kCW / kGroup)];
      s2[r] = make_float2(sb.x, sb.x);
      b2[r] = make_float2(sb.y, sb.y);
    }
    float2 P[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) P[r][mm] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      float2 xv[MT][kCPW / 2];
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int j = 0; j < kCPW / 4; ++j) {
          const float4 t = *reinterpret_cast<const float4*>(
              xl + mm * xs_m + (i * (kCW / 4) + wi * (kCPW / 4) + j) * 128);
          xv[mm][2 * j] = make_float2(t.x, t.y);
          xv[mm][2 * j + 1] = make_float2(t.z, t.w);
        }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t word = wi == 0 ? cw[r].x : wi == 1 ? cw[r].y : wi == 2 ? cw[r].z : cw[r].w;
        float2 f[kCPW / 2];
        U::run(word, f);
#pragma unroll
        for (int mm = 0; mm < MT; ++mm)
#pragma unroll
          for (int j = 0; j < kCPW / 2; ++j) P[r][mm] = __ffma2_rn(f[j], xv[mm][j], P[r][mm]);
      }
    }
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) {
      const float2 X = xsl[mm * xsum_m + i * 32];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float2 D = __ffma2_rn(neg_magic, X, P[r][mm]);
        acc[r][mm] = __ffma2_rn(s2[r], D, acc[r][mm]);
        acc[r][mm] = __ffma2_rn(b2[r], X, acc[r][mm]);
      }
    }
  }
}

// The warp-wide sums of the R x MT accumulators.  Lane l ends with value
// index vi = l / (32 / (R*MT)), i.e. row vi / MT and token vi % MT of the
// warp's rows; the first lane of each such run is the one that stores it.
template <int MT, int R>
struct RowSums {
  static constexpr int kV = R * MT;
  static constexpr int kLanesPerValue = 32 / kV;
  static __device__ __forceinline__ int value_index(int lane) { return lane / kLanesPerValue; }
  static __device__ __forceinline__ bool owner(int lane) { return lane % kLanesPerValue == 0; }
  static __device__ __forceinline__ float reduce(float2 (&acc)[R][MT], int lane) {
    float v[kV];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) v[r * MT + mm] = acc[r][mm].x + acc[r][mm].y;
    return butterfly_sum<kV>(v, lane);
  }
};

// Store one finished sum: a linear layer's bias joins the f32 sum before the
// one rounding (or the f32 value is stored as it is).
template <typename AT>
__device__ __forceinline__ void store_value(float total, int row, int m, void* __restrict__ y,
                                            int64_t ldy, const AT* __restrict__ layer_bias,
                                            bool y_f32) {
  if (layer_bias) total += Act<AT>::to_f32(layer_bias[row]);
  if (y_f32)
    static_cast<float*>(y)[int64_t(m) * ldy + row] = total;
  else
    static_cast<AT*>(y)[int64_t(m) * ldy + row] = Act<AT>::from_f32_rn(total);
}

// Reduce the warp's R x MT sums across lanes and store them (row-major y with
// leading dimension ldy).  Returns true on the lanes that stored a value.
template <int MT, int R, typename AT>
__device__ __forceinline__ bool store_rows(float2 (&acc)[R][MT], int lane, int row0, int m0,
                                           int N, int M, void* __restrict__ y, int64_t ldy,
                                           const AT* __restrict__ layer_bias, bool y_f32) {
  using RS = RowSums<MT, R>;
  const float total = RS::reduce(acc, lane);
  const int vi = RS::value_index(lane);
  const int row = row0 + vi / MT, m = m0 + vi % MT;
  if (RS::owner(lane) && row < N && m < M) {
    store_value<AT>(total, row, m, y, ldy, layer_bias, y_f32);
    return true;
  }
  return false;
}

template <int MT, int R, typename AT>
__device__ __forceinline__ bool store_rows(float2 (&acc)[R][MT], int lane, int row0, int m0,
                                           int N, int M, AT* __restrict__ y, int64_t ldy) {
  return store_rows<MT, R, AT>(acc, lane, row0, m0, N, M, static_cast<void*>(y), ldy,
                               static_cast<const AT*>(nullptr), false);
}

}  // namespace qmvcore
}  // namespace qlin
