// qmv: fused dequantise-into-matvec on CUDA cores for decode (small M).
//
// y[m][n] = sum_k x[m][k] * (q[n][k]*scale[n][g(k)] + bias[n][g(k)])
//
// The packed payload is streamed from HBM exactly once per M-tile with 128-bit
// non-caching loads, unpacked in registers and consumed immediately: the
// reconstructed weight never exists outside registers ("track(upstream-iree):
// fused dequant->matmul for the packed int8 bandwidth win", section "The
// blocker (measured)": materialising it is what made the unfused path slower
// than f16).  Any N >= 1 works, including N not a multiple of 4 ("Metal
// backend: import qmv_impl from MLX").
//
// Arithmetic (f32 throughout, one RNE to the output type at the end):
//   A 16-byte chunk of a row holds CW = 128/bits codes that all share one
//   group (64 % CW == 0).  Each code is turned into the float MAGIC + q by
//   OR-ing it into the mantissa of MAGIC (128 for 4-bit, 256 for 8-bit: the
//   code lands on the unit bit, so the value is exact).  Per chunk
//       P = sum_k x_k * (MAGIC + q_k)          (packed f32x2 FMAs)
//       sum_k x_k * w_hat_k = scale * (P - MAGIC * X) + bias * X,
//   with X = sum_k x_k over the chunk, computed once per CTA and shared by all
//   rows.  MAGIC is within a factor 10-20 of the codes, so the cancellation in
//   P - MAGIC*X costs ~4-5 bits of the 24: far inside the output tolerance.
//
// Work split: a CTA of 8 warps owns RG*R consecutive rows (RG row groups of R
// rows); the KS = 8/RG warps of a row group split the chunks of those rows,
// lanes taking consecutive 16-byte chunks (coalesced 512-byte warp reads).
// Partial sums are reduced with warp shuffles, then across the KS warps in
// shared memory; no global workspace is used.

#include <algorithm>

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int BITS>
struct Unpack;

// 4-bit: nibble pairs are spread to bytes, then each byte is placed in bits
// 16..23 under the exponent of 128.0f (0x43000000) with one byte permute.
template <>
struct Unpack<4> {
  static constexpr int kCodes = 8;  // per word
  static constexpr float kMagic = 128.0f;
  static __device__ __forceinline__ void run(uint32_t w, float2 (&f)[4]) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // codes 0,2,4,6 in bytes 0..3
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // codes 1,3,5,7
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t sel = 0x7054u | (uint32_t(i) << 8);
      f[i].x = u32_as_f32(__byte_perm(lo, 0x43000000u, sel));
      f[i].y = u32_as_f32(__byte_perm(hi, 0x43000000u, sel));
    }
  }
};

// 8-bit: each byte is shifted to bits 15..22 under the exponent of 256.0f
// (0x43800000), whose unit bit is bit 15.
template <>
struct Unpack<8> {
  static constexpr int kCodes = 4;
  static constexpr float kMagic = 256.0f;
  static __device__ __forceinline__ void run(uint32_t w, float2 (&f)[2]) {
    constexpr uint32_t kM = 0x007F8000u, kE = 0x43800000u;
    f[0].x = u32_as_f32(((w << 15) & kM) | kE);
    f[0].y = u32_as_f32(((w << 7) & kM) | kE);
    f[1].x = u32_as_f32(((w >> 1) & kM) | kE);
    f[1].y = u32_as_f32(((w >> 9) & kM) | kE);
  }
};

template <int BITS, int MT, int R, typename AT>
__global__ void __launch_bounds__(kThreads) qmv_kernel(
    const AT* __restrict__ x, const uint32_t* __restrict__ wq, const AT* __restrict__ scales,
    const AT* __restrict__ biases, AT* __restrict__ y, int M, int N, int K, int ks_log2) {
  using U = Unpack<BITS>;
  constexpr int kCW = 128 / BITS;          // codes per 16-byte chunk
  constexpr int kCPW = U::kCodes;          // codes per word
  extern __shared__ float4 smem4[];
  float* xs = reinterpret_cast<float*>(smem4);  // [MT][K]
  const int C = K / kCW;                        // chunks per row
  float* xc = xs + MT * K;                      // [MT][C] chunk sums
  const int ksplit = 1 << ks_log2;
  const int rg_count = kWarps >> ks_log2;
  float* red = xc + MT * C;                     // [ksplit][rg_count*R*MT]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ks = warp & (ksplit - 1), rg = warp >> ks_log2;
  const int rows_per_cta = rg_count * R;
  const int row_base = blockIdx.x * rows_per_cta;
  const int m0 = blockIdx.y * MT;

  // ---- stage x (as f32) and its per-chunk sums in shared memory
  for (int i = tid; i < MT * (K / 8); i += kThreads) {
    const int mm = i / (K / 8), k8 = i % (K / 8);
    float v[8];
    if (m0 + mm < M) {
      const uint4 raw = *reinterpret_cast<const uint4*>(x + int64_t(m0 + mm) * K + k8 * 8);
      const AT* h = reinterpret_cast<const AT*>(&raw);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = Act<AT>::to_f32(h[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    float4* dst = reinterpret_cast<float4*>(xs + mm * K + k8 * 8);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __syncthreads();
  for (int i = tid; i < MT * C; i += kThreads) {
    const int mm = i / C, c = i % C;
    const float* src = xs + mm * K + c * kCW;
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < kCW; ++j) s += src[j];
    xc[i] = s;
  }
  __syncthreads();

  // ---- main loop over this warp's chunks
  const int64_t wpr = int64_t(K) * BITS / 32;  // words per row
  const int gpr = K / kGroup;                   // groups per row
  const int row0 = row_base + rg * R;
  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) acc[r][mm] = 0.0f;

  for (int c = ks * 32 + lane; c < C; c += 32 * ksplit) {
    uint4 wv[R];
    float sv[R], bv[R];
    const int g = (c * kCW) / kGroup;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = min(row0 + r, N - 1);
      wv[r] = ldg_nc_v4(wq + int64_t(row) * wpr + 4 * c);
      sv[r] = Act<AT>::to_f32(scales[int64_t(row) * gpr + g]);
      bv[r] = Act<AT>::to_f32(biases[int64_t(row) * gpr + g]);
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
      for (int mm = 0; mm < MT; ++mm) {
        const float4* src = reinterpret_cast<const float4*>(xs + mm * K + c * kCW + wi * kCPW);
#pragma unroll
        for (int j = 0; j < kCPW / 4; ++j) {
          const float4 t = src[j];
          xv[mm][2 * j] = make_float2(t.x, t.y);
          xv[mm][2 * j + 1] = make_float2(t.z, t.w);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t word = (&wv[r].x)[wi];
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
      const float X = xc[mm * C + c];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float p = P[r][mm].x + P[r][mm].y;
        acc[r][mm] = __fmaf_rn(sv[r], __fmaf_rn(-U::kMagic, X, p), acc[r][mm]);
        acc[r][mm] = __fmaf_rn(bv[r], X, acc[r][mm]);
      }
    }
  }

  // ---- reduce: lanes, then the KS warps of the row group
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int mm = 0; mm < MT; ++mm) {
      float v = acc[r][mm];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[ks * (rows_per_cta * MT) + (rg * R + r) * MT + mm] = v;
    }
  __syncthreads();
  for (int i = tid; i < rows_per_cta * MT; i += kThreads) {
    const int mm = i / rows_per_cta, rr = i % rows_per_cta;
    const int row = row_base + rr, m = m0 + mm;
    if (row >= N || m >= M) continue;
    float s = 0.0f;
    for (int k2 = 0; k2 < ksplit; ++k2) s += red[k2 * (rows_per_cta * MT) + rr * MT + mm];
    y[int64_t(m) * N + row] = Act<AT>::from_f32_rn(s);
  }
}

size_t smem_bytes(int MT, int R, int K, int bits, int ks_log2) {
  const int C = K * bits / 128;
  const int rows = (kWarps >> ks_log2) * R;
  return size_t(4) * (size_t(MT) * K + size_t(MT) * C + size_t(1 << ks_log2) * rows * MT);
}

template <int BITS, int MT, int R, typename AT>
qlin_status launch_t(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, int ks_log2, cudaStream_t st) {
  auto kern = qmv_kernel<BITS, MT, R, AT>;
  const size_t smem = smem_bytes(MT, R, int(K), BITS, ks_log2);
  static int attr_set_for = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_for != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
        cudaSuccess)
      return check_launch("qmv: cudaFuncSetAttribute");
    attr_set_for = dev;
  }
  const int rows_per_cta = (kWarps >> ks_log2) * R;
  dim3 grid(unsigned((N + rows_per_cta - 1) / rows_per_cta), unsigned((M + MT - 1) / MT));
  kern<<<grid, kThreads, smem, st>>>(static_cast<const AT*>(x), wq,
                                     static_cast<const AT*>(scales),
                                     static_cast<const AT*>(biases), static_cast<AT*>(y), int(M),
                                     int(N), int(K), ks_log2);
  return check_launch("qmv_kernel");
}

template <int BITS, int MT, typename AT>
qlin_status pick_r(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                   void* y, int64_t M, int64_t N, int64_t K, int ks_log2, cudaStream_t st) {
  // Fewest rows per thread that still gives every SM a few CTAs: fewer rows
  // per CTA spread small N over more SMs.
  const int64_t want = int64_t(sm_count()) * 3;
  const int64_t tiles_m = (M + MT - 1) / MT;
  const int rg = kWarps >> ks_log2;
  auto ctas = [&](int R) { return ((N + rg * R - 1) / (rg * R)) * tiles_m; };
  if (ctas(4) >= want)
    return launch_t<BITS, MT, 4, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
  if (ctas(2) >= want)
    return launch_t<BITS, MT, 2, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
  return launch_t<BITS, MT, 1, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
}

template <int BITS, typename AT>
qlin_status dispatch(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  const int64_t C = K * BITS / 128;
  int ks_log2 = 0;
  while (ks_log2 < 3 && (int64_t(32) << (ks_log2 + 1)) <= C) ++ks_log2;
  int MT = M >= 3 ? 4 : int(M);
  while (MT > 1 && smem_bytes(MT, 4, int(K), BITS, ks_log2) > 160 * 1024) MT >>= 1;
  if (smem_bytes(MT, 4, int(K), BITS, ks_log2) > 200 * 1024)
    return fail(QLIN_ERR_UNSUPPORTED, "qlin_qmv: K=%lld too large for the staged x", (long long)K);
  switch (MT) {
    case 1: return pick_r<BITS, 1, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
    case 2: return pick_r<BITS, 2, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
    default: return pick_r<BITS, 4, AT>(x, wq, scales, biases, y, M, N, K, ks_log2, st);
  }
}

}  // namespace

qlin_status launch_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                       void* y, int64_t M, int64_t N, int64_t K, int bits, qlin_dtype dtype,
                       cudaStream_t st) {
  if (dtype == QLIN_F16)
    return bits == 4 ? dispatch<4, __half>(x, wq, scales, biases, y, M, N, K, st)
                     : dispatch<8, __half>(x, wq, scales, biases, y, M, N, K, st);
  return bits == 4 ? dispatch<4, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, st)
                   : dispatch<8, __nv_bfloat16>(x, wq, scales, biases, y, M, N, K, st);
}

}  // namespace qlin
