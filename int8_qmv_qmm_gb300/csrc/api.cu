// Public C entry points of libqlin: argument validation, then dispatch to the
// launchers.  Nothing is launched unless every check passes.

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "qlin_internal.h"
#include "qlin_testing.h"

namespace qlin {

static thread_local char g_last_error[512] = "";

qlin_status fail(qlin_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

qlin_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(QLIN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return QLIN_OK;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qlin_status check_format(int64_t N, int64_t K, int bits, int group_size) {
  if (bits != 4 && bits != 8) return fail(QLIN_ERR_UNSUPPORTED, "bits=%d (supported: 4, 8)", bits);
  if (group_size != kGroup)
    return fail(QLIN_ERR_UNSUPPORTED, "group_size=%d (supported: 64)", group_size);
  if (N < 0) return fail(QLIN_ERR_INVALID_ARG, "N=%lld < 0", (long long)N);
  if (K <= 0 || K % group_size)
    return fail(QLIN_ERR_INVALID_ARG, "K=%lld must be a positive multiple of group_size=%d",
                (long long)K, group_size);
  if (N > (int64_t(1) << 31) || K > (int64_t(1) << 24))
    return fail(QLIN_ERR_UNSUPPORTED, "N=%lld or K=%lld beyond the supported range",
                (long long)N, (long long)K);
  return QLIN_OK;
}

qlin_status check_act_dtype(qlin_dtype d, const char* what) {
  if (d != QLIN_F16 && d != QLIN_BF16)
    return fail(QLIN_ERR_UNSUPPORTED, "%s dtype %d (supported: QLIN_F16, QLIN_BF16)", what, (int)d);
  return QLIN_OK;
}

using MatmulLauncher = qlin_status (*)(const void*, const uint32_t*, const void*, const void*,
                                       void*, int64_t, int64_t, int64_t, int, qlin_dtype,
                                       unsigned, const Epilogue&, cudaStream_t);

const Epilogue kPlainEpilogue = {nullptr, 0};

qlin_status matmul_entry(const char* name, MatmulLauncher launch, const void* x,
                         const uint32_t* wq, const void* scales, const void* biases, void* y,
                         int64_t M, int64_t N, int64_t K, int bits, int group_size,
                         qlin_dtype dtype, unsigned flags, void* stream,
                         const Epilogue& ep = kPlainEpilogue) {
  qlin_status s = check_format(N, K, bits, group_size);
  if (s != QLIN_OK) return s;
  if (flags & ~unsigned(QLIN_OVERLAP_PREVIOUS))
    return fail(QLIN_ERR_INVALID_ARG, "%s: unknown flags 0x%x", name, flags);
  if ((s = check_act_dtype(dtype, "activation/scale")) != QLIN_OK) return s;
  if (M < 0) return fail(QLIN_ERR_INVALID_ARG, "%s: M=%lld < 0", name, (long long)M);
  if (M > (int64_t(1) << 31)) return fail(QLIN_ERR_UNSUPPORTED, "%s: M too large", name);
  if (M == 0 || N == 0) return QLIN_OK;  // empty product: nothing to write
  if (!x || !wq || !scales || !biases || !y)
    return fail(QLIN_ERR_INVALID_ARG, "%s: null pointer argument", name);
  if (!aligned(x, 16) || !aligned(wq, 16))
    return fail(QLIN_ERR_MISALIGNED, "%s: x and wq must be 16-byte aligned", name);
  if (!aligned(scales, 2) || !aligned(biases, 2) || !aligned(y, ep.y_f32 ? 4 : 2))
    return fail(QLIN_ERR_MISALIGNED,
                "%s: scales and biases must be 2-byte aligned, y %d-byte aligned", name,
                ep.y_f32 ? 4 : 2);
  if (ep.bias && !aligned(ep.bias, 2))
    return fail(QLIN_ERR_MISALIGNED, "%s: the layer bias must be 2-byte aligned", name);
  return launch(x, wq, scales, biases, y, M, N, K, bits, dtype, flags, ep,
                reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace qlin

using namespace qlin;

extern "C" {

const char* qlin_status_str(qlin_status s) {
  switch (s) {
    case QLIN_OK: return "QLIN_OK";
    case QLIN_ERR_INVALID_ARG: return "QLIN_ERR_INVALID_ARG";
    case QLIN_ERR_UNSUPPORTED: return "QLIN_ERR_UNSUPPORTED";
    case QLIN_ERR_MISALIGNED: return "QLIN_ERR_MISALIGNED";
    case QLIN_ERR_CUDA: return "QLIN_ERR_CUDA";
    case QLIN_ERR_DEVICE_TIMEOUT: return "QLIN_ERR_DEVICE_TIMEOUT";
  }
  return "QLIN_ERR_UNKNOWN";
}

const char* qlin_last_error(void) { return g_last_error; }

int qlin_version(void) { return 100; }

qlin_status qlin_quantize_affine(const float* w, int64_t N, int64_t K, int bits, int group_size,
                                 qlin_dtype sdtype, uint32_t* wq, void* scales, void* biases,
                                 void* stream) {
  g_last_error[0] = 0;
  qlin_status s = check_format(N, K, bits, group_size);
  if (s != QLIN_OK) return s;
  if ((s = check_act_dtype(sdtype, "scale")) != QLIN_OK) return s;
  if (N == 0) return QLIN_OK;
  if (!w || !wq || !scales || !biases)
    return fail(QLIN_ERR_INVALID_ARG, "qlin_quantize_affine: null pointer argument");
  if (!aligned(w, 16) || !aligned(wq, 16))
    return fail(QLIN_ERR_MISALIGNED, "qlin_quantize_affine: w and wq must be 16-byte aligned");
  if (!aligned(scales, 2) || !aligned(biases, 2))
    return fail(QLIN_ERR_MISALIGNED, "qlin_quantize_affine: scales/biases must be 2-byte aligned");
  return launch_quantize(w, N, K, bits, sdtype, wq, scales, biases,
                         reinterpret_cast<cudaStream_t>(stream));
}

qlin_status qlin_dequant(const uint32_t* wq, const void* scales, const void* biases, int64_t N,
                         int64_t K, int bits, int group_size, qlin_dtype sdtype,
                         qlin_dtype out_dtype, void* w_out, void* stream) {
  g_last_error[0] = 0;
  qlin_status s = check_format(N, K, bits, group_size);
  if (s != QLIN_OK) return s;
  if ((s = check_act_dtype(sdtype, "scale")) != QLIN_OK) return s;
  if (out_dtype != QLIN_F32 && out_dtype != sdtype)
    return fail(QLIN_ERR_UNSUPPORTED,
                "qlin_dequant: out_dtype must be QLIN_F32 or the scale dtype (%d)", (int)sdtype);
  if (N == 0) return QLIN_OK;
  if (!wq || !scales || !biases || !w_out)
    return fail(QLIN_ERR_INVALID_ARG, "qlin_dequant: null pointer argument");
  if (!aligned(wq, 16) || !aligned(w_out, 16))
    return fail(QLIN_ERR_MISALIGNED, "qlin_dequant: wq and w_out must be 16-byte aligned");
  if (!aligned(scales, 2) || !aligned(biases, 2))
    return fail(QLIN_ERR_MISALIGNED, "qlin_dequant: scales/biases must be 2-byte aligned");
  return launch_dequant(wq, scales, biases, N, K, bits, sdtype, out_dtype, w_out,
                        reinterpret_cast<cudaStream_t>(stream));
}

qlin_status qlin_qmv(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                     qlin_dtype dtype, void* stream) {
  g_last_error[0] = 0;
  return matmul_entry("qlin_qmv", launch_qmv, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, 0u, stream);
}

qlin_status qlin_qmv_ex(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                        void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                        qlin_dtype dtype, unsigned flags, void* stream) {
  g_last_error[0] = 0;
  return matmul_entry("qlin_qmv_ex", launch_qmv, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, flags, stream);
}

qlin_status qlin_qmm_ex(const void* x, const uint32_t* wq, const void* scales,
                        const void* biases, void* y, int64_t M, int64_t N, int64_t K, int bits,
                        int group_size, qlin_dtype dtype, unsigned flags, void* stream) {
  g_last_error[0] = 0;
  return matmul_entry("qlin_qmm_ex", launch_qmm, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, flags, stream);
}

qlin_status qlin_qmm(const void* x, const uint32_t* wq, const void* scales, const void* biases,
                     void* y, int64_t M, int64_t N, int64_t K, int bits, int group_size,
                     qlin_dtype dtype, void* stream) {
  g_last_error[0] = 0;
  return matmul_entry("qlin_qmm", launch_qmm, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, 0u, stream);
}

size_t qlin_qmv_chain_workspace_size(int n_links) {
  if (n_links <= 0) return 0;
  return (size_t(n_links) * sizeof(unsigned) + 255) / 256 * 256;
}

}  // extern "C"

namespace qlin {
namespace {
qlin_status chain_entry(const void* x0, const qlin_link* links, int n_links, int bits,
                        int group_size, qlin_dtype dtype, void* workspace, size_t workspace_bytes,
                        const ChainWaitOptions& wo, void* stream) {
  if (!links || n_links < 1 || n_links > chain_max_links())
    return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: need 1..%d links", chain_max_links());
  qlin_status s = check_act_dtype(dtype, "activation/scale");
  if (s != QLIN_OK) return s;
  if (!workspace || workspace_bytes < qlin_qmv_chain_workspace_size(n_links))
    return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: workspace of %zu bytes needed",
                qlin_qmv_chain_workspace_size(n_links));
  if (!aligned(workspace, 16))
    return fail(QLIN_ERR_MISALIGNED, "qlin_qmv_chain: workspace must be 16-byte aligned");
  for (int l = 0; l < n_links; ++l) {
    const qlin_link& L = links[l];
    if ((s = check_format(L.N, L.K, bits, group_size)) != QLIN_OK)
      return fail(s, "qlin_qmv_chain: link %d: %s", l, qlin_last_error());
    if (L.N < 1 || L.N > (int64_t(1) << 30) || L.K > (int64_t(1) << 20))
      return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: link %d: N=%lld K=%lld out of range", l,
                  (long long)L.N, (long long)L.K);
    if (!L.wq || !L.scales || !L.biases || !L.y)
      return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: link %d: null pointer", l);
    if (!aligned(L.wq, 16) || !aligned(L.scales, 2) || !aligned(L.biases, 2) || !aligned(L.y, 2))
      return fail(QLIN_ERR_MISALIGNED, "qlin_qmv_chain: link %d: misaligned pointer", l);
    if (L.input < 0) {
      if (L.input != -1) return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: link %d: input", l);
      if (!x0) return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: link %d reads a null x0", l);
      if (!aligned(x0, 16))
        return fail(QLIN_ERR_MISALIGNED, "qlin_qmv_chain: x0 must be 16-byte aligned");
    } else {
      if (L.input >= l)
        return fail(QLIN_ERR_INVALID_ARG, "qlin_qmv_chain: link %d reads link %d (not earlier)",
                    l, L.input);
      const qlin_link& D = links[L.input];
      if (L.input_offset < 0 || int64_t(L.input_offset) + L.K > D.N)
        return fail(QLIN_ERR_INVALID_ARG,
                    "qlin_qmv_chain: link %d reads past the end of link %d's output", l, L.input);
      if (!aligned(static_cast<const uint8_t*>(D.y) + int64_t(L.input_offset) * 2, 16))
        return fail(QLIN_ERR_MISALIGNED,
                    "qlin_qmv_chain: link %d's input must start 16-byte aligned", l);
    }
  }
  return launch_qmv_chain(x0, links, n_links, bits, dtype, workspace, wo,
                          reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace
}  // namespace qlin

extern "C" {

qlin_status qlin_qmv_chain(const void* x0, const qlin_link* links, int n_links, int bits,
                           int group_size, qlin_dtype dtype, void* workspace,
                           size_t workspace_bytes, void* stream) {
  g_last_error[0] = 0;
  return chain_entry(x0, links, n_links, bits, group_size, dtype, workspace, workspace_bytes,
                     kDefaultChainWaits, stream);
}

int qlin_testing_qmv_split(int64_t N, int64_t K, int bits, int sm_count) {
  if ((bits != 4 && bits != 8) || K < 64 || K % 64 != 0 || N < 1 || sm_count < 1) return -1;
  return qlin::qmv_plan_split(N, K, bits, sm_count);
}

qlin_status qlin_testing_qmv_chain_stalled(const void* x0, const qlin_link* links, int n_links,
                                           int bits, int group_size, qlin_dtype dtype,
                                           void* workspace, size_t workspace_bytes,
                                           int stalled_link, unsigned wait_limit_us,
                                           void* stream) {
  g_last_error[0] = 0;
  if (!links || n_links < 1 || stalled_link < 0 || stalled_link >= n_links)
    return fail(QLIN_ERR_INVALID_ARG, "qlin_testing_qmv_chain_stalled: stalled_link %d",
                stalled_link);
  bool read = false;
  for (int l = stalled_link + 1; l < n_links; ++l) read = read || links[l].input == stalled_link;
  if (!read)
    return fail(QLIN_ERR_INVALID_ARG,
                "qlin_testing_qmv_chain_stalled: no link reads link %d, nothing would wait",
                stalled_link);
  if (wait_limit_us < 1 || wait_limit_us > 2000000u)
    return fail(QLIN_ERR_INVALID_ARG, "qlin_testing_qmv_chain_stalled: wait_limit_us %u",
                wait_limit_us);
  const ChainWaitOptions wo = {1000ull * wait_limit_us, stalled_link};
  return chain_entry(x0, links, n_links, bits, group_size, dtype, workspace, workspace_bytes, wo,
                     stream);
}

int64_t qlin_crossover_m_dtype(int64_t N, int64_t K, int bits, qlin_dtype dtype) {
  (void)bits;
  // QLIN_CROSSOVER_M (a positive integer) overrides the measured choice; read
  // once, on the first call
  static const long long env_m = [] {
    const char* env = getenv("QLIN_CROSSOVER_M");
    const long long v = env && *env ? atoll(env) : 0;
    return v >= 1 ? v : 0;
  }();
  if (env_m) return env_m;
  // Measured on GB300 (batched decode, M = 2..16, weights rotated over 2.5x
  // the L2 size; 4- and 8-bit alike, f16 and bf16).  qmv streams the weights
  // once per tile of 4 tokens, so its time steps up at M = 5, 9, ...; qmm's
  // stays flat for M <= 256.  On the larger matrices (N*K >= 6.3 M: 3072 x
  // 2048, 8192 x 2048, 2048 x 8192) qmm is the faster from M = 5 (8192 x 2048,
  // 8-bit f16, M = 6: 12.3 vs 16.1 us), and with f16 already at M = 4 when
  // K > N (2048 x 8192: 17.7 vs 18.2 us).  On 2048 x 2048, where qmm has only
  // 16 row tiles to spread, qmv stays the faster up to M = 8 (bf16, M = 8: 9.2
  // vs 11.3 us; M = 12: 11.9 vs 11.3 us).
  if (dtype == QLIN_F16 && K > N) return 4;
  return N * K >= int64_t(6) * 1024 * 1024 ? 5 : 9;
}

int64_t qlin_crossover_m(int64_t N, int64_t K, int bits) {
  return qlin_crossover_m_dtype(N, K, bits, QLIN_F16);
}

qlin_status qlin_linear(const void* x, const uint32_t* wq, const void* scales,
                        const void* biases, void* y, int64_t M, int64_t N, int64_t K, int bits,
                        int group_size, qlin_dtype dtype, void* stream) {
  g_last_error[0] = 0;
  if (M < qlin_crossover_m_dtype(N, K, bits, dtype))
    return matmul_entry("qlin_linear", launch_qmv, x, wq, scales, biases, y, M, N, K, bits,
                        group_size, dtype, 0u, stream);
  return matmul_entry("qlin_linear", launch_qmm, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, 0u, stream);
}

qlin_status qlin_linear_ex(const void* x, const uint32_t* wq, const void* scales,
                           const void* biases, const void* layer_bias, void* y, int64_t M,
                           int64_t N, int64_t K, int bits, int group_size, qlin_dtype dtype,
                           qlin_dtype y_dtype, void* stream) {
  g_last_error[0] = 0;
  if (y_dtype != QLIN_F32 && y_dtype != dtype)
    return fail(QLIN_ERR_UNSUPPORTED,
                "qlin_linear_ex: y dtype %d must be float32 or the activation dtype %d",
                int(y_dtype), int(dtype));
  const Epilogue ep = {layer_bias, y_dtype == QLIN_F32 ? 1 : 0};
  if (M < qlin_crossover_m_dtype(N, K, bits, dtype))
    return matmul_entry("qlin_linear_ex", launch_qmv, x, wq, scales, biases, y, M, N, K, bits,
                        group_size, dtype, 0u, stream, ep);
  return matmul_entry("qlin_linear_ex", launch_qmm, x, wq, scales, biases, y, M, N, K, bits,
                      group_size, dtype, 0u, stream, ep);
}

qlin_status qlin_device_status(int* flags) {
  g_last_error[0] = 0;
  if (!flags) return fail(QLIN_ERR_INVALID_ARG, "qlin_device_status: null pointer");
  unsigned fm = 0, fv = 0, fc = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = qmm_take_device_status(&fm);
  if (e == cudaSuccess) e = qmv_take_device_status(&fv);
  if (e == cudaSuccess) e = chain_take_device_status(&fc);
  if (e != cudaSuccess)
    return fail(QLIN_ERR_CUDA, "qlin_device_status: %s", cudaGetErrorString(e));
  // qmm waits in the low byte, qmv waits in the next one, the chain above
  *flags = static_cast<int>((fm & 0xffu) | ((fv & 0xffu) << 8) | ((fc & 0xffu) << 16));
  return QLIN_OK;
}

}  // extern "C"
