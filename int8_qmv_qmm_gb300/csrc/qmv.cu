// qmv: fused dequantise-into-matvec on CUDA cores for decode (small M).
//
// y[m][n] = sum_k x[m][k] * (q[n][k]*scale[n][g(k)] + bias[n][g(k)])
//
// The packed payload is streamed from HBM exactly once per M-tile and consumed
// straight out of shared memory: the reconstructed weight never exists outside
// registers ("track(upstream-iree): fused dequant->matmul for the packed int8
// bandwidth win", section "The blocker (measured)": materialising it is what
// made the unfused path slower than f16).  Any N >= 1 works, including N not a
// multiple of 4 ("Metal backend: import qmv_impl from MLX").
//
// Data movement.  A CTA owns row blocks of RB = 8*R consecutive rows
// (persistent: block b, b + grid, ...).  A block is cut into k-tiles of KT
// bytes per row; one (block, k-tile) is one pipeline stage.  A producer warp
// fills a ring of shared-memory stages with 1-D bulk async copies (one per
// row, so no register holds in-flight data and each CTA keeps S stages --
// 50-100 KB -- in flight), and, when scales/biases are 16-byte aligned per
// row slice, bulk-copies their slices too (otherwise the consumers read them
// from global memory).  Eight consumer warps compute.  The producer starts
// before the kernel waits for its predecessor on the stream, so with
// programmatic dependent launch the weights stream while the previous kernel
// finishes.
//
// Arithmetic (f32 throughout, one RNE to the output type at the end):
//   A 16-byte chunk of a row holds CW = 128/bits codes sharing one group
//   (64 % CW == 0).  Each code becomes the float MAGIC + q by placing it under
//   the exponent of MAGIC (4-bit: 128.0f, code bits 16..19; 8-bit: 32768.0f,
//   code bits 8..15): one byte permute per code, exact.  Per chunk, with
//   f32x2 FMAs over (even, odd) code positions,
//       P = sum_k x_k * (MAGIC + q_k),   X = sum_k x_k
//       sum_k x_k * w_hat_k = scale * (P - MAGIC * X) + bias * X.
//   X (split even/odd) is computed once per CTA and shared by all rows.  The
//   cancellation in P - MAGIC*X costs log2(MAGIC / mean code) bits of the 24
//   (about 4 for 4-bit, 8 for 8-bit), far inside the output tolerance.
//
// x is staged once per CTA as f32 in a lane-transposed layout
// ([round][4-code group][lane][4]) so that lanes reading consecutive 16-byte
// chunks of a row read consecutive 16-byte words of x: conflict-free.  Warp w
// computes rows w*R .. w*R+R-1 of each stage; lanes take consecutive chunks.
// Per-lane sums of a block's R*MT outputs are reduced across lanes with a
// halving butterfly after the block's last k-tile.  No global workspace.
//
// Every mbarrier wait is bounded; a wait that gives up sets a device status
// bit and the CTA unwinds after its outstanding copies have landed.

#include <algorithm>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "sm100_ptx.cuh"

namespace qlin {

__device__ unsigned int g_qmv_status = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kProducerWarp = kConsumerWarps;

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

struct Shape {
  int M, N, K;
  int C;            // 16-byte chunks per row
  int rounds;       // ceil(C / 32): rounds of the lane-transposed x layout
  int kt_bytes;     // bytes of one row per k-tile (multiple of 16, divides the row)
  int n_kt;         // k-tiles per row
  int n_blocks;     // row blocks
  int stages;       // ring depth
  int stage_bytes;  // bytes of one stage (weights, then scales and biases)
  unsigned flags;
};

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <int BITS, int MT, int R, typename AT, bool SCALE_COPY>
__global__ void __launch_bounds__(kThreads) qmv_kernel(
    const AT* __restrict__ x, const uint32_t* __restrict__ wq, const AT* __restrict__ scales,
    const AT* __restrict__ biases, AT* __restrict__ y, const Shape sh) {
  using U = Unpack<BITS>;
  constexpr int kCW = 128 / BITS;  // codes per 16-byte chunk
  constexpr int kCPW = U::kCodes;  // codes per word
  constexpr int kRB = kConsumerWarps * R;
  constexpr int kV = R * MT;
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = sh.K, N = sh.N, C = sh.C;
  const int row_bytes = K * BITS / 8;
  const int gpr = K / kGroup;
  const int kt_chunks = sh.kt_bytes / 16;
  const int kt_groups = sh.kt_bytes * (8 / BITS) / kGroup;  // groups per row per k-tile
  const int xs_m = sh.rounds * 32 * kCW;  // floats per row of x in the transposed layout

  // shared memory: [stages][stage_bytes] | x (f32) | xsum (f32x2) | barriers
  uint8_t* ring = smem;
  float* xs = reinterpret_cast<float*>(ring + size_t(sh.stages) * sh.stage_bytes);
  float2* xsum = reinterpret_cast<float2*>(xs + MT * xs_m);
  uint64_t* bars = reinterpret_cast<uint64_t*>(xsum + MT * sh.rounds * 32);
  const uint32_t ring_u32 = ptx::smem_u32(ring);
  const uint32_t full0 = ptx::smem_u32(bars), empty0 = full0 + 8u * sh.stages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int m0 = blockIdx.y * MT;

  if (tid == 0) {
    for (int s = 0; s < sh.stages; ++s) {
      ptx::mbar_init(full0 + 8u * s, 1);
      ptx::mbar_init(empty0 + 8u * s, kConsumerWarps);
    }
    ptx::fence_mbar_init();
  }
  __syncthreads();

  // stage units of this CTA: blocks blockIdx.x, +gridDim.x, ...; k-tiles in order
  const int n_my_blocks =
      sh.n_blocks > int(blockIdx.x) ? (sh.n_blocks - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                                    : 0;
  const int n_units = n_my_blocks * sh.n_kt;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int u = 0;
    bool ok = true;
    for (; u < n_units; ++u) {
      const int s = u % sh.stages;
      const uint32_t round = uint32_t(u / sh.stages);
      if (u >= sh.stages && !ptx::mbar_wait(empty0 + 8u * s, (round - 1) & 1u)) {
        if (lane == 0) atomicOr(&g_qmv_status, 1u);
        ok = false;
        break;
      }
      const int blk = int(blockIdx.x) + (u / sh.n_kt) * int(gridDim.x), kt = u % sh.n_kt;
      const int row0 = blk * kRB;
      const int nr = min(kRB, N - row0);
      const uint32_t w_bytes = uint32_t(sh.kt_bytes);
      const uint32_t sb_bytes = SCALE_COPY ? uint32_t(kt_groups * 2) : 0u;
      const uint32_t stage = ring_u32 + uint32_t(s) * uint32_t(sh.stage_bytes);
      if (lane == 0)
        ptx::mbar_arrive_expect_tx(full0 + 8u * s, uint32_t(nr) * (w_bytes + 2 * sb_bytes));
      __syncwarp();
      if (sh.n_kt == 1) {
        // whole rows: the block is one contiguous range (and so are its
        // scales and biases)
        if (lane == 0) {
          bulk_copy(stage, reinterpret_cast<const uint8_t*>(wq) + int64_t(row0) * row_bytes,
                    uint32_t(nr) * w_bytes, full0 + 8u * s);
          if constexpr (SCALE_COPY) {
            const uint32_t sb0 = stage + uint32_t(kRB) * w_bytes;
            const int64_t g0 = int64_t(row0) * gpr;
            bulk_copy(sb0, scales + g0, uint32_t(nr) * sb_bytes, full0 + 8u * s);
            bulk_copy(sb0 + uint32_t(kRB) * sb_bytes, biases + g0, uint32_t(nr) * sb_bytes,
                      full0 + 8u * s);
          }
        }
        continue;
      }
      for (int r = lane; r < nr; r += 32) {
        const int row = row0 + r;
        bulk_copy(stage + uint32_t(r) * w_bytes,
                  reinterpret_cast<const uint8_t*>(wq) + int64_t(row) * row_bytes +
                      int64_t(kt) * sh.kt_bytes,
                  w_bytes, full0 + 8u * s);
        if constexpr (SCALE_COPY) {
          const int64_t g0 = int64_t(row) * gpr + int64_t(kt) * kt_groups;
          const uint32_t sb0 = stage + uint32_t(kRB) * w_bytes;
          bulk_copy(sb0 + uint32_t(r) * sb_bytes, scales + g0, sb_bytes, full0 + 8u * s);
          bulk_copy(sb0 + uint32_t(kRB) * sb_bytes + uint32_t(r) * sb_bytes, biases + g0,
                    sb_bytes, full0 + 8u * s);
        }
      }
    }
    if (!ok) {
      // let the copies already issued land before the CTA's memory goes away
      const int first = u > sh.stages ? u - sh.stages : 0;
      for (int v = first; v < u; ++v)
        if (!ptx::mbar_wait(full0 + 8u * (v % sh.stages), uint32_t(v / sh.stages) & 1u))
          if (lane == 0) atomicOr(&g_qmv_status, 16u);
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  // x is produced by the preceding kernel: wait for it (a no-op unless this is
  // a programmatic dependent launch), then let the next kernel launch early.
  grid_dependency_wait();
  grid_launch_dependents();
  for (int e = tid; e < MT * (K / 8); e += kConsumerWarps * 32) {
    const int mm = e / (K / 8), k0 = (e % (K / 8)) * 8;
    float v[8];
    if (m0 + mm < sh.M) {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + int64_t(m0 + mm) * K + k0);
      const AT* h = reinterpret_cast<const AT*>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = Act<AT>::to_f32(h[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    const int c = k0 / kCW, j4 = (k0 % kCW) / 4;
    float* base = xs + mm * xs_m + ((c >> 5) * (kCW / 4) * 32 + (c & 31)) * 4;
    *reinterpret_cast<float4*>(base + j4 * 128) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(base + (j4 + 1) * 128) = make_float4(v[4], v[5], v[6], v[7]);
  }
  consumers_sync();
  for (int e = tid; e < MT * sh.rounds * 32; e += kConsumerWarps * 32) {
    const int mm = e / (sh.rounds * 32), c = e % (sh.rounds * 32);
    float2 s = make_float2(0.0f, 0.0f);
    if (c < C) {
      const float* base = xs + mm * xs_m + ((c >> 5) * (kCW / 4) * 32 + (c & 31)) * 4;
#pragma unroll
      for (int j4 = 0; j4 < kCW / 4; ++j4) {
        const float4 t = *reinterpret_cast<const float4*>(base + j4 * 128);
        s.x += t.x + t.z;
        s.y += t.y + t.w;
      }
    }
    xsum[e] = s;
  }
  consumers_sync();

  const float2 neg_magic = make_float2(-U::kMagic, -U::kMagic);
  float2 acc[R][MT];
  for (int u = 0; u < n_units; ++u) {
    const int s = u % sh.stages;
    const int blk = int(blockIdx.x) + (u / sh.n_kt) * int(gridDim.x), kt = u % sh.n_kt;
    const int rb0 = blk * kRB + warp * R;  // this warp's first row
    if (kt == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) acc[r][mm] = make_float2(0.0f, 0.0f);
    }
    if (!ptx::mbar_wait(full0 + 8u * s, uint32_t(u / sh.stages) & 1u)) {
      if (lane == 0) atomicOr(&g_qmv_status, 2u);
      break;
    }
    const uint8_t* stage = ring + size_t(s) * sh.stage_bytes;
    const uint8_t* wst = stage + size_t(warp * R) * sh.kt_bytes;
    const AT* sst = reinterpret_cast<const AT*>(stage + size_t(kRB) * sh.kt_bytes);
    const AT* bst = sst + kRB * kt_groups;
    for (int cl = lane; cl < kt_chunks; cl += 32) {
      const int c = kt * kt_chunks + cl;   // chunk index within the row
      const int gl = (cl * kCW) / kGroup;  // group within the k-tile
      uint4 cw[R];
      float2 s2[R], b2[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        // rows past N were not copied: their values are never stored
        cw[r] = *reinterpret_cast<const uint4*>(wst + size_t(r) * sh.kt_bytes + cl * 16);
        float sv, bv;
        if constexpr (SCALE_COPY) {
          sv = Act<AT>::to_f32(sst[(warp * R + r) * kt_groups + gl]);
          bv = Act<AT>::to_f32(bst[(warp * R + r) * kt_groups + gl]);
        } else {
          const int64_t gi = int64_t(min(rb0 + r, N - 1)) * gpr + (c * kCW) / kGroup;
          sv = Act<AT>::to_f32(scales[gi]);
          bv = Act<AT>::to_f32(biases[gi]);
        }
        s2[r] = make_float2(sv, sv);
        b2[r] = make_float2(bv, bv);
      }
      const float* xbase = xs + ((c >> 5) * (kCW / 4) * 32 + (c & 31)) * 4;
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
                xbase + mm * xs_m + (wi * (kCPW / 4) + j) * 128);
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
        const float2 X = xsum[mm * sh.rounds * 32 + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float2 D = __ffma2_rn(neg_magic, X, P[r][mm]);
          acc[r][mm] = __ffma2_rn(s2[r], D, acc[r][mm]);
          acc[r][mm] = __ffma2_rn(b2[r], X, acc[r][mm]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(empty0 + 8u * s);

    if (kt == sh.n_kt - 1) {
      float v[kV];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int mm = 0; mm < MT; ++mm) v[r * MT + mm] = acc[r][mm].x + acc[r][mm].y;
      const float total = butterfly_sum<kV>(v, lane);
      constexpr int kLanesPerValue = 32 / kV;
      const int vi = lane / kLanesPerValue;
      const int row = rb0 + vi / MT, m = m0 + vi % MT;
      if ((lane % kLanesPerValue) == 0 && row < N && m < sh.M)
        y[int64_t(m) * N + row] = Act<AT>::from_f32_rn(total);
    }
  }
}

// ------------------------------------------------------------------- host
size_t smem_for(const Shape& sh, int MT, int bits) {
  const int cw = 128 / bits;
  return size_t(sh.stages) * sh.stage_bytes + size_t(MT) * sh.rounds * 32 * cw * 4 +
         size_t(MT) * sh.rounds * 32 * 8 + size_t(sh.stages) * 16;
}

template <int BITS, int MT, int R, typename AT, bool SC>
qlin_status launch_t(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, const Shape& sh, size_t smem, cudaStream_t st) {
  auto kern = qmv_kernel<BITS, MT, R, AT, SC>;
  // per device: attribute set once; occupancy cached per dynamic smem size
  static int attr_dev = -1;
  static size_t occ_smem[8] = {0};
  static int occ_blocks[8] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return check_launch("qmv: cudaFuncSetAttribute");
    for (int i = 0; i < 8; ++i) occ_smem[i] = 0;
    attr_dev = dev;
  }
  int blocks_per_sm = 0;
  for (int i = 0; i < 8 && !blocks_per_sm; ++i)
    if (occ_smem[i] == smem) blocks_per_sm = occ_blocks[i];
  if (!blocks_per_sm) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, smem) != cudaSuccess ||
        b < 1)
      b = 1;
    blocks_per_sm = b;
    int slot = 0;
    while (slot < 7 && occ_smem[slot]) ++slot;
    occ_smem[slot] = smem;
    occ_blocks[slot] = b;
  }
  const int64_t m_tiles = (sh.M + MT - 1) / MT;
  if (m_tiles > 65535) return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv: M too large");
  const int64_t resident = int64_t(blocks_per_sm) * sm_count();
  const int64_t per_tile = std::max<int64_t>(1, resident / std::min<int64_t>(m_tiles, resident));
  const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(sh.n_blocks, per_tile));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(gx), unsigned(m_tiles), 1u);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (sh.flags & QLIN_OVERLAP_PREVIOUS) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const AT*>(x), wq,
                                           static_cast<const AT*>(scales),
                                           static_cast<const AT*>(biases), static_cast<AT*>(y),
                                           sh);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QLIN_ERR_CUDA, "qmv_kernel launch: %s", cudaGetErrorString(e));
  }
  return check_launch("qmv_kernel");
}

template <int BITS, int MT, typename AT>
qlin_status dispatch_mt(const void* x, const uint32_t* wq, const void* scales,
                        const void* biases, void* y, Shape sh, cudaStream_t st) {
  const int64_t sms = sm_count();
  const int row_bytes = sh.K * BITS / 8;
  const int gpr = sh.K / kGroup;
  // rows per consumer warp: more rows (x reuse, fewer blocks) when rows are
  // plentiful, fewer when the launch would otherwise leave SMs idle
  int R = sh.N >= 32 * 4 * sms ? 4 : sh.N >= 16 * 2 * sms ? 2 : 1;
  if (MT >= 4 && R > 2) R = 2;
  const int RB = kConsumerWarps * R;
  // k-tile: stages of about 32 KB of weights: the whole row when it fits,
  // else the smallest split into equal 16-byte-multiple tiles that does
  const int kt_max = std::max(512, 32768 / RB);
  int n_kt = 1;
  while (row_bytes / n_kt > kt_max || row_bytes % n_kt || (row_bytes / n_kt) % 16) ++n_kt;
  sh.n_kt = n_kt;
  sh.kt_bytes = row_bytes / n_kt;
  const int kt_codes = sh.kt_bytes * (8 / BITS);
  const int kt_groups = kt_codes / kGroup;
  const bool scale_copy = kt_codes % kGroup == 0 && (kt_groups * 2) % 16 == 0 &&
                          (gpr * 2) % 16 == 0 &&
                          (reinterpret_cast<uintptr_t>(scales) % 16) == 0 &&
                          (reinterpret_cast<uintptr_t>(biases) % 16) == 0;
  sh.stage_bytes = RB * sh.kt_bytes + (scale_copy ? 2 * RB * kt_groups * 2 : 0);
  sh.stage_bytes = (sh.stage_bytes + 127) / 128 * 128;
  sh.n_blocks = (sh.N + RB - 1) / RB;
  // ring depth: about 96 KB of stages, so that two CTAs fit on an SM
  sh.stages = std::max(2, std::min(8, (96 * 1024) / sh.stage_bytes));
  size_t smem = smem_for(sh, MT, BITS);
  while (sh.stages > 2 && smem > 110 * 1024) {
    --sh.stages;
    smem = smem_for(sh, MT, BITS);
  }
  if (smem > 220 * 1024)
    return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv: K=%d too large for the staged x", sh.K);
#define QLIN_QMV_LAUNCH(RR)                                                                 \
  return scale_copy                                                                         \
             ? launch_t<BITS, MT, RR, AT, true>(x, wq, scales, biases, y, sh, smem, st)     \
             : launch_t<BITS, MT, RR, AT, false>(x, wq, scales, biases, y, sh, smem, st)
  switch (R) {
    case 4: QLIN_QMV_LAUNCH(4);
    case 2: QLIN_QMV_LAUNCH(2);
    default: QLIN_QMV_LAUNCH(1);
  }
#undef QLIN_QMV_LAUNCH
}

template <int BITS, typename AT>
qlin_status dispatch(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, unsigned flags, cudaStream_t st) {
  Shape sh{};
  sh.flags = flags;
  sh.M = int(M);
  sh.N = int(N);
  sh.K = int(K);
  sh.C = int(K * BITS / 128);
  sh.rounds = (sh.C + 31) / 32;
  const int MT = M >= 3 ? 4 : int(M);
  switch (MT) {
    case 1: return dispatch_mt<BITS, 1, AT>(x, wq, scales, biases, y, sh, st);
    case 2: return dispatch_mt<BITS, 2, AT>(x, wq, scales, biases, y, sh, st);
    default: return dispatch_mt<BITS, 4, AT>(x, wq, scales, biases, y, sh, st);
  }
}

}  // namespace

qlin_status launch_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       unsigned flags, cudaStream_t st) {
  if (dtype == QLIN_F16)
    return bits == 4 ? dispatch<4, __half>(x, wq, scales, biases, y, M, N, K, flags, st)
                     : dispatch<8, __half>(x, wq, scales, biases, y, M, N, K, flags, st);
  return bits == 4 ? dispatch<4, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, flags, st)
                   : dispatch<8, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, flags, st);
}

cudaError_t qmv_take_device_status(unsigned* flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_qmv_status, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_qmv_status, &zero, sizeof(zero));
  *flags = v;
  return e;
}

}  // namespace qlin
