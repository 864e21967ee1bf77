// The C ABI: argument checks on the host, then the launches.  Nothing here computes
// any part of the path; every result comes from the kernels.
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cmath>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace pgq {

namespace {
constexpr unsigned long long WAIT_LIMIT_DEFAULT_NS = 2000000000ull;   // 2 s
std::atomic<unsigned long long> g_wait_limit_ns{WAIT_LIMIT_DEFAULT_NS};
std::atomic<int> g_stall{0};
thread_local char g_err[512] = "";
std::mutex g_dev_mu;
DeviceInfo g_dev[64];
bool g_dev_ok[64];
bool g_dev_done[64];
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int stall_injected() { return g_stall.load(std::memory_order_relaxed); }

int set_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

bool device_info(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_done[dev]) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    bool ok = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    ok = ok && cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess;
    ok = ok && cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess;
    ok = ok && cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess;
    d.smem_optin = (size_t)v;
    g_dev[dev] = d;
    g_dev_ok[dev] = ok && d.cc_major == 10 && d.cc_minor == 3;
    g_dev_done[dev] = true;
  }
  *out = g_dev[dev];
  return g_dev_ok[dev];
}

}  // namespace pgq

using namespace pgq;

#define REQUIRE(cond, status, ...)                \
  do {                                            \
    if (!(cond)) return set_error(status, __VA_ARGS__); \
  } while (0)

#define GET_DEVICE(dev)                                                                  \
  DeviceInfo dev;                                                                        \
  if (!device_info(&dev)) return set_error(PGQ_ENODEV, "no current compute-capability-10.3 device")

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

extern "C" {

const char* pgq_status_string(int status) {
  switch (status) {
    case PGQ_OK: return "ok";
    case PGQ_EINVAL: return "invalid argument";
    case PGQ_EALIGN: return "misaligned pointer";
    case PGQ_EUNSUPPORTED: return "shape outside the kernels' limits";
    case PGQ_ECUDA: return "CUDA error";
    case PGQ_ETIMEOUT: return "device-side wait expired";
    case PGQ_ENODEV: return "no compute-capability-10.3 device";
    case PGQ_EWORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

const char* pgq_last_error(void) { return g_err; }

int pgq_abi_version(void) { return 1; }

int pgq_device_check(void) {
  GET_DEVICE(dev);
  return PGQ_OK;
}

int pgq_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) ns = WAIT_LIMIT_DEFAULT_NS;
  REQUIRE(ns >= 1000ull && ns <= 60000000000ull, PGQ_EINVAL, "set_wait_limit_ns: %llu ns outside 1 us .. 60 s", ns);
  g_wait_limit_ns.store(ns);
  return PGQ_OK;
}

unsigned long long pgq_wait_limit_ns(void) { return wait_limit_ns(); }

int pgq_debug_stall(int on) {
  REQUIRE(on == 0 || on == 1, PGQ_EINVAL, "debug_stall: %d is neither 0 nor 1", on);
  g_stall.store(on);
  return PGQ_OK;
}

int pgq_last_device_status(const void* workspace, void* stream) {
  GET_DEVICE(dev);
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_status(e);
  int dec = PGQ_OK;
  const int rc = decode_status_read_and_clear(&dec);
  if (rc) return rc;
  int ws[2] = {PGQ_OK, PGQ_OK};
  if (workspace) {
    char* st = const_cast<char*>(static_cast<const char*>(workspace)) + prefill_status_offset();
    e = cudaMemcpy(ws, st, sizeof(ws), cudaMemcpyDeviceToHost);
    // read and clear: a later call on the workspace starts from a clean record
    if (e == cudaSuccess && (ws[0] != PGQ_OK || ws[1] != PGQ_OK)) e = cudaMemset(st, 0, sizeof(ws));
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (dec != PGQ_OK) return dec;
  return ws[0] != PGQ_OK ? ws[0] : ws[1];
}


int pgq_add_rmsnorm(float* h, const float* add, const float* gamma, float eps, int B, int n, float* y,
                    float* inv_rms, void* stream) {
  REQUIRE(h && gamma && y, PGQ_EINVAL, "add_rmsnorm: h, gamma and y must be non-null");
  REQUIRE(B >= 1 && B <= 65535, PGQ_EINVAL, "add_rmsnorm: B=%d outside 1..65535", B);
  REQUIRE(n >= 4 && n <= (1 << 20) && n % 4 == 0, PGQ_EINVAL, "add_rmsnorm: n=%d must be a multiple of 4 in 4..2^20", n);
  REQUIRE(eps >= 0.f, PGQ_EINVAL, "add_rmsnorm: eps must be >= 0");
  REQUIRE(aligned16(h) && aligned16(gamma) && aligned16(y) && (!add || aligned16(add)), PGQ_EALIGN,
          "add_rmsnorm: h, add, gamma, y must be 16-byte aligned");
  REQUIRE(!inv_rms || aligned4(inv_rms), PGQ_EALIGN, "add_rmsnorm: inv_rms must be 4-byte aligned");
  const size_t bytes = (size_t)B * n * sizeof(float);
  REQUIRE(!overlaps(y, bytes, h, bytes) && (!add || !overlaps(y, bytes, add, bytes)), PGQ_EINVAL,
          "add_rmsnorm: y must not overlap h or add");
  GET_DEVICE(dev);
  return launch_add_rmsnorm(h, add, gamma, eps, 0.f, 0, B, n, y, inv_rms, as_stream(stream));
}

int pgq_add_rmsnorm_ex(float* h, const float* add, const float* gamma, float eps, float scale, int flags, int B, int n,
                       float* y, float* inv_rms, void* stream) {
  REQUIRE((flags & ~PGQ_NORM_GEMMA) == 0, PGQ_EINVAL, "add_rmsnorm_ex: unknown flags 0x%x", flags);
  REQUIRE(scale == scale && scale != INFINITY && scale != -INFINITY, PGQ_EINVAL, "add_rmsnorm_ex: scale must be finite");
  REQUIRE(h && gamma && y, PGQ_EINVAL, "add_rmsnorm_ex: h, gamma and y must be non-null");
  REQUIRE(B >= 1 && B <= 65535, PGQ_EINVAL, "add_rmsnorm_ex: B=%d outside 1..65535", B);
  REQUIRE(n >= 4 && n <= (1 << 20) && n % 4 == 0, PGQ_EINVAL, "add_rmsnorm_ex: n=%d must be a multiple of 4 in 4..2^20",
          n);
  REQUIRE(eps >= 0.f, PGQ_EINVAL, "add_rmsnorm_ex: eps must be >= 0");
  REQUIRE(aligned16(h) && aligned16(gamma) && aligned16(y) && (!add || aligned16(add)), PGQ_EALIGN,
          "add_rmsnorm_ex: h, add, gamma, y must be 16-byte aligned");
  REQUIRE(!inv_rms || aligned4(inv_rms), PGQ_EALIGN, "add_rmsnorm_ex: inv_rms must be 4-byte aligned");
  const size_t bytes = (size_t)B * n * sizeof(float);
  REQUIRE(!overlaps(y, bytes, h, bytes) && (!add || !overlaps(y, bytes, add, bytes)), PGQ_EINVAL,
          "add_rmsnorm_ex: y must not overlap h or add");
  GET_DEVICE(dev);
  return launch_add_rmsnorm(h, add, gamma, eps, scale, (flags & PGQ_NORM_GEMMA) ? 1 : 0, B, n, y, inv_rms,
                            as_stream(stream));
}

int pgq_sandwich_rmsnorm(const float* x, const float* w1, float* h, const float* w2, float eps, float scale, int flags,
                         int B, int n, float* out, float* mid, float* inv1, float* inv2, void* stream) {
  REQUIRE((flags & ~PGQ_NORM_GEMMA) == 0, PGQ_EINVAL, "sandwich_rmsnorm: unknown flags 0x%x", flags);
  REQUIRE(scale == scale && scale != INFINITY && scale != -INFINITY, PGQ_EINVAL,
          "sandwich_rmsnorm: scale must be finite");
  REQUIRE(x && w1 && h && w2 && out, PGQ_EINVAL, "sandwich_rmsnorm: x, w1, h, w2 and out must be non-null");
  REQUIRE(B >= 1 && B <= 65535, PGQ_EINVAL, "sandwich_rmsnorm: B=%d outside 1..65535", B);
  REQUIRE(n >= 4 && n <= PGQ_SANDWICH_NMAX && n % 4 == 0, PGQ_EINVAL,
          "sandwich_rmsnorm: n=%d must be a multiple of 4 in 4..%d", n, PGQ_SANDWICH_NMAX);
  REQUIRE(eps >= 0.f, PGQ_EINVAL, "sandwich_rmsnorm: eps must be >= 0");
  REQUIRE(aligned16(x) && aligned16(w1) && aligned16(h) && aligned16(w2) && aligned16(out) && (!mid || aligned16(mid)),
          PGQ_EALIGN, "sandwich_rmsnorm: x, w1, h, w2, out and mid must be 16-byte aligned");
  REQUIRE((!inv1 || aligned4(inv1)) && (!inv2 || aligned4(inv2)), PGQ_EALIGN, "sandwich_rmsnorm: inv1/inv2 4-byte");
  const size_t bytes = (size_t)B * n * sizeof(float);
  REQUIRE(!overlaps(out, bytes, h, bytes) && !overlaps(out, bytes, x, bytes) && !overlaps(h, bytes, x, bytes),
          PGQ_EINVAL, "sandwich_rmsnorm: x, h and out must not overlap");
  REQUIRE(!mid || (!overlaps(mid, bytes, x, bytes) && !overlaps(mid, bytes, h, bytes) && !overlaps(mid, bytes, out, bytes)),
          PGQ_EINVAL, "sandwich_rmsnorm: mid must not overlap x, h or out");
  GET_DEVICE(dev);
  return launch_sandwich(x, w1, h, w2, eps, scale, (flags & PGQ_NORM_GEMMA) ? 1 : 0, B, n, out, mid, inv1, inv2, dev,
                         as_stream(stream));
}

int pgq_relu2(float* v, size_t n, void* stream) {
  if (n == 0) return PGQ_OK;
  REQUIRE(v, PGQ_EINVAL, "relu2: v must be non-null");
  REQUIRE(aligned16(v), PGQ_EALIGN, "relu2: v must be 16-byte aligned");
  GET_DEVICE(dev);
  return launch_relu2(v, n, as_stream(stream), dev.sms);
}

int pgq_argmax(const float* logits, int B, int V, int32_t* ids, void* stream) {
  REQUIRE(logits && ids, PGQ_EINVAL, "argmax: logits and ids must be non-null");
  REQUIRE(B >= 1 && B <= 65535 && V >= 1, PGQ_EINVAL, "argmax: B=%d V=%d out of range", B, V);
  REQUIRE(aligned4(logits) && aligned4(ids), PGQ_EALIGN, "argmax: pointers must be 4-byte aligned");
  GET_DEVICE(dev);
  return launch_argmax(logits, B, V, ids, as_stream(stream));
}

// ------------------------------------------------------------------ decode GEMVs
static int check_decode_common(const char* name, int rows, int cols, const float* x, int B, const float* gamma,
                               float eps, const float* y_or_null, int epilogue, const float* residual) {
  REQUIRE(x, PGQ_EINVAL, "%s: x must be non-null", name);
  REQUIRE(rows >= 1, PGQ_EINVAL, "%s: rows=%d must be >= 1", name, rows);
  REQUIRE(cols >= 32 && cols % 32 == 0, PGQ_EINVAL, "%s: cols=%d must be a positive multiple of 32", name, cols);
  REQUIRE(B >= 1 && B <= PGQ_DECODE_BMAX, PGQ_EINVAL, "%s: B=%d outside 1..%d", name, B, PGQ_DECODE_BMAX);
  REQUIRE((size_t)B * cols <= PGQ_STAGE_MAX, PGQ_EUNSUPPORTED, "%s: B*cols=%d exceeds %d staged values", name,
          B * cols, PGQ_STAGE_MAX);
  REQUIRE(epilogue >= PGQ_EPI_NONE && epilogue <= PGQ_EPI_ADD, PGQ_EINVAL, "%s: bad epilogue %d", name, epilogue);
  REQUIRE(epilogue != PGQ_EPI_ADD || residual, PGQ_EINVAL, "%s: PGQ_EPI_ADD needs a residual", name);
  REQUIRE(!gamma || eps >= 0.f, PGQ_EINVAL, "%s: eps must be >= 0", name);
  REQUIRE(aligned16(x) && (!gamma || aligned16(gamma)), PGQ_EALIGN, "%s: x and gamma must be 16-byte aligned", name);
  REQUIRE((!y_or_null || aligned4(y_or_null)) && (!residual || aligned4(residual)), PGQ_EALIGN,
          "%s: y and residual must be 4-byte aligned", name);
  if (y_or_null) {
    const size_t yb = (size_t)B * rows * sizeof(float);
    REQUIRE(!overlaps(y_or_null, yb, x, (size_t)B * cols * sizeof(float)), PGQ_EINVAL, "%s: y overlaps x", name);
    REQUIRE(!residual || residual == y_or_null || !overlaps(y_or_null, yb, residual, yb), PGQ_EINVAL,
            "%s: residual must be y itself or not overlap it", name);
  }
  return PGQ_OK;
}

namespace {
// (build_only != NULL: check the arguments and fill *build_only instead of launching)
int gemv_f16_impl(const uint16_t* W, int rows, int cols, const float* x, int B, const float* gamma, float eps, float* y,
                  int epilogue, const float* residual, int early_weights, void* stream, GvParams* build_only = nullptr);
}  // namespace

int pgq_gemv_f16(const uint16_t* W, int rows, int cols, const float* x, int B, const float* gamma, float eps, float* y,
                 int epilogue, const float* residual, void* stream) {
  return gemv_f16_impl(W, rows, cols, x, B, gamma, eps, y, epilogue, residual, 0, stream);
}

namespace {
// pgq_gemv_f16 with the early-weights flag (GvParams::early_weights)
int gemv_f16_impl(const uint16_t* W, int rows, int cols, const float* x, int B, const float* gamma, float eps, float* y,
                  int epilogue, const float* residual, int early_weights, void* stream, GvParams* build_only) {
  REQUIRE(W && y, PGQ_EINVAL, "gemv_f16: W and y must be non-null");
  REQUIRE(aligned16(W), PGQ_EALIGN, "gemv_f16: W must be 16-byte aligned");
  int st = check_decode_common("gemv_f16", rows, cols, x, B, gamma, eps, y, epilogue, residual);
  if (st) return st;
  GET_DEVICE(dev);
  GvParams P{};
  P.job[0] = GvJob{reinterpret_cast<const uint8_t*>(W), nullptr, y, residual, rows, 0, epilogue, 0};
  P.in[0] = GvInput{x, gamma};
  P.njobs = 1;
  P.ninputs = 1;
  P.B = B;
  P.cols = cols;
  P.eps = eps;
  P.early_weights = early_weights;
  if (build_only) {
    *build_only = P;
    return PGQ_OK;
  }
  return launch_gemv(P, false, false, dev, as_stream(stream));
}
}  // namespace

size_t pgq_argmax_workspace_bytes(int B) {
  DeviceInfo dev;
  if (!device_info(&dev)) dev.sms = 160;  // an upper bound when no device is current
  if (B < 1) B = 1;
  return gemv_argmax_workspace_bytes(B, dev);
}

int pgq_gemv_f16_argmax(const uint16_t* W, int rows, int cols, const float* x, int B, const float* gamma, float eps,
                        float* logits, int32_t* ids, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(W && ids, PGQ_EINVAL, "gemv_f16_argmax: W and ids must be non-null");
  REQUIRE(aligned16(W) && aligned4(ids), PGQ_EALIGN, "gemv_f16_argmax: W 16-byte, ids 4-byte aligned");
  int st = check_decode_common("gemv_f16_argmax", rows, cols, x, B, gamma, eps, logits, PGQ_EPI_NONE, nullptr);
  if (st) return st;
  GET_DEVICE(dev);
  const size_t need = gemv_argmax_workspace_bytes(B, dev);
  REQUIRE(workspace && aligned16(workspace) && workspace_bytes >= need, PGQ_EWORKSPACE,
          "gemv_f16_argmax: workspace needs %zu bytes, 16-byte aligned", need);
  GvParams P{};
  P.job[0] = GvJob{reinterpret_cast<const uint8_t*>(W), nullptr, logits, nullptr, rows, 0, PGQ_EPI_NONE, 0};
  P.in[0] = GvInput{x, gamma};
  P.njobs = 1;
  P.ninputs = 1;
  P.B = B;
  P.cols = cols;
  P.eps = eps;
  const size_t parts = (size_t)dev.sms * B;
  char* ws = static_cast<char*>(workspace);
  P.part_val = reinterpret_cast<float*>(ws);
  P.part_idx = reinterpret_cast<int*>(ws + ((parts * sizeof(float) + 15) & ~size_t(15)));
  P.ticket = reinterpret_cast<unsigned*>(ws + ((parts * sizeof(float) + 15) & ~size_t(15)) +
                                         ((parts * sizeof(int) + 15) & ~size_t(15)));
  P.ids = ids;
  return launch_gemv(P, false, true, dev, as_stream(stream));
}

int pgq_gemv_f16_argmax_static(const uint16_t* W, int rows, int cols, const float* x, int B, const float* gamma,
                               float eps, float* logits, int32_t* ids, void* stream) {
  REQUIRE(B >= 1 && B <= PGQ_DECODE_BMAX, PGQ_EINVAL, "gemv_f16_argmax_static: B=%d outside 1..%d", B,
          PGQ_DECODE_BMAX);
  GET_DEVICE(dev);
  const size_t need = gemv_argmax_workspace_bytes(B, dev);
  REQUIRE(need <= PGQ_STATIC_SCRATCH_BYTES, PGQ_EUNSUPPORTED,
          "gemv_f16_argmax_static: %d SMs x B=%d need %zu bytes of scratch, more than the fixed %d", dev.sms, B, need,
          PGQ_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  const int st = argmax_static_scratch(&scratch, &scratch_bytes);
  if (st) return st;
  return pgq_gemv_f16_argmax(W, rows, cols, x, B, gamma, eps, logits, ids, scratch, scratch_bytes, stream);
}

int pgq_gemv_q8(const int8_t* codes, const uint16_t* params, int rows, int cols, const float* x, int B,
                const float* gamma, float eps, float* y, int epilogue, const float* residual, void* stream) {
  pgq_q8_job job{codes, params, rows, 0, y, epilogue, residual};
  pgq_input in{x, gamma};
  return pgq_gemv_q8_multi(&job, 1, &in, 1, cols, B, eps, stream);
}

namespace {
// pgq_gemv_q8_multi with the early-weights flag (GvParams::early_weights); with
// build_only != NULL it checks the arguments and fills *build_only instead of launching
int gemv_q8_multi_impl(const pgq_q8_job* jobs, int njobs, const pgq_input* inputs, int ninputs, int cols, int B,
                       float eps, int early_weights, void* stream, GvParams* build_only = nullptr);
}  // namespace

int pgq_gemv_q8_multi(const pgq_q8_job* jobs, int njobs, const pgq_input* inputs, int ninputs, int cols, int B,
                      float eps, void* stream) {
  return gemv_q8_multi_impl(jobs, njobs, inputs, ninputs, cols, B, eps, 0, stream);
}

namespace {
int gemv_q8_multi_impl(const pgq_q8_job* jobs, int njobs, const pgq_input* inputs, int ninputs, int cols, int B,
                       float eps, int early_weights, void* stream, GvParams* build_only) {
  REQUIRE(jobs && inputs, PGQ_EINVAL, "gemv_q8: jobs and inputs must be non-null");
  REQUIRE(njobs >= 1 && njobs <= PGQ_MULTI_MAX, PGQ_EINVAL, "gemv_q8: njobs=%d outside 1..%d", njobs, PGQ_MULTI_MAX);
  REQUIRE(ninputs >= 1 && ninputs <= MAX_INPUTS, PGQ_EINVAL, "gemv_q8: ninputs=%d outside 1..%d", ninputs,
          MAX_INPUTS);
  REQUIRE((size_t)ninputs * B * cols <= PGQ_STAGE_MAX, PGQ_EUNSUPPORTED,
          "gemv_q8: ninputs*B*cols=%d exceeds %d staged values", ninputs * B * cols, PGQ_STAGE_MAX);
  for (int i = 0; i < ninputs; ++i) {
    int st = check_decode_common("gemv_q8", 1, cols, inputs[i].x, B, inputs[i].gamma, eps, nullptr, PGQ_EPI_NONE,
                                 nullptr);
    if (st) return st;
  }
  GvParams P{};
  for (int j = 0; j < njobs; ++j) {
    const pgq_q8_job& J = jobs[j];
    REQUIRE(J.codes && J.params && J.y, PGQ_EINVAL, "gemv_q8: job %d has a null codes/params/y", j);
    REQUIRE(aligned8(J.codes) && aligned4(J.params), PGQ_EALIGN, "gemv_q8: job %d codes 8-byte, params 4-byte", j);
    REQUIRE(J.input >= 0 && J.input < ninputs, PGQ_EINVAL, "gemv_q8: job %d input %d out of range", j, J.input);
    int st = check_decode_common("gemv_q8", J.rows, cols, inputs[J.input].x, B, inputs[J.input].gamma, eps, J.y,
                                 J.epilogue, J.residual);
    if (st) return st;
    for (int i = 0; i < ninputs; ++i)
      REQUIRE(!overlaps(J.y, (size_t)B * J.rows * 4, inputs[i].x, (size_t)B * cols * 4), PGQ_EINVAL,
              "gemv_q8: job %d output overlaps input %d", j, i);
    P.job[j] = GvJob{reinterpret_cast<const uint8_t*>(J.codes), reinterpret_cast<const uint32_t*>(J.params), J.y,
                     J.residual, J.rows, J.input, J.epilogue, 0};
  }
  GET_DEVICE(dev);
  for (int i = 0; i < ninputs; ++i) P.in[i] = GvInput{inputs[i].x, inputs[i].gamma};
  P.njobs = njobs;
  P.ninputs = ninputs;
  P.B = B;
  P.cols = cols;
  P.eps = eps;
  P.early_weights = early_weights;
  if (build_only) {
    *build_only = P;
    return PGQ_OK;
  }
  return launch_gemv(P, true, false, dev, as_stream(stream));
}
}  // namespace

// ------------------------------------------------------------------ q8_2f decode
namespace {
// One launch of q8_2f projections sharing cols and B (the TMA decode kernel only).
struct Q82Job {
  const int8_t* codes;
  const uint16_t* rs;
  const uint16_t* cf;
  int rows, input;
  float* y;
  int epilogue;
  const float* residual;
};
int gemv_q82f_multi_impl(const Q82Job* jobs, int njobs, const pgq_input* inputs, int ninputs, int cols, int B,
                         float eps, int early_weights, void* stream) {
  REQUIRE(njobs >= 1 && njobs <= PGQ_MULTI_MAX && ninputs >= 1 && ninputs <= MAX_INPUTS, PGQ_EINVAL,
          "gemv_q82f: %d jobs, %d inputs", njobs, ninputs);
  REQUIRE((size_t)ninputs * B * cols <= PGQ_STAGE_MAX, PGQ_EUNSUPPORTED,
          "gemv_q82f: ninputs*B*cols=%d exceeds %d staged values", ninputs * B * cols, PGQ_STAGE_MAX);
  for (int i = 0; i < ninputs; ++i) {
    int st = check_decode_common("gemv_q82f", 1, cols, inputs[i].x, B, inputs[i].gamma, eps, nullptr, PGQ_EPI_NONE,
                                 nullptr);
    if (st) return st;
  }
  GvParams P{};
  for (int j = 0; j < njobs; ++j) {
    const Q82Job& J = jobs[j];
    REQUIRE(J.codes && J.rs && J.cf && J.y, PGQ_EINVAL, "gemv_q82f: job %d has a null codes/row_scale/col_field/y", j);
    REQUIRE(aligned16(J.codes) && aligned16(J.cf) && (reinterpret_cast<uintptr_t>(J.rs) & 1) == 0, PGQ_EALIGN,
            "gemv_q82f: job %d codes and col_field 16-byte, row_scale 2-byte aligned", j);
    REQUIRE(J.input >= 0 && J.input < ninputs, PGQ_EINVAL, "gemv_q82f: job %d input %d out of range", j, J.input);
    int st = check_decode_common("gemv_q82f", J.rows, cols, inputs[J.input].x, B, inputs[J.input].gamma, eps, J.y,
                                 J.epilogue, J.residual);
    if (st) return st;
    for (int i = 0; i < ninputs; ++i)
      REQUIRE(!overlaps(J.y, (size_t)B * J.rows * 4, inputs[i].x, (size_t)B * cols * 4), PGQ_EINVAL,
              "gemv_q82f: job %d output overlaps input %d", j, i);
    GvJob g{};
    g.w = reinterpret_cast<const uint8_t*>(J.codes);
    g.y = J.y;
    g.residual = J.residual;
    g.rows = J.rows;
    g.input = J.input;
    g.epilogue = J.epilogue;
    g.rs = J.rs;
    g.cf = J.cf;
    P.job[j] = g;
  }
  GET_DEVICE(dev);
  for (int i = 0; i < ninputs; ++i) P.in[i] = GvInput{inputs[i].x, inputs[i].gamma};
  P.njobs = njobs;
  P.ninputs = ninputs;
  P.B = B;
  P.cols = cols;
  P.eps = eps;
  P.early_weights = early_weights;
  P.q82f = 1;
  return launch_gemv(P, true, false, dev, as_stream(stream));
}
}  // namespace

int pgq_gemv_q82f(const int8_t* codes, const uint16_t* row_scale, const uint16_t* col_field, int rows, int cols,
                  const float* x, int B, const float* gamma, float eps, float* y, int epilogue, const float* residual,
                  void* stream) {
  const Q82Job job{codes, row_scale, col_field, rows, 0, y, epilogue, residual};
  const pgq_input in{x, gamma};
  return gemv_q82f_multi_impl(&job, 1, &in, 1, cols, B, eps, 0, stream);
}

int pgq_q82f_decode_layer(const pgq_q82f_layer* L, const float* x, const float* x_o, const float* gamma, float eps,
                          float* q, float* k, float* v, float* o, float* u, float* down, int flags, void* stream) {
  REQUIRE(L && x && x_o && gamma && q && k && v && o && u && down, PGQ_EINVAL, "q82f_decode_layer: null pointer");
  REQUIRE((flags & ~PGQ_WEIGHTS_STABLE) == 0, PGQ_EINVAL, "q82f_decode_layer: unknown flags 0x%x", flags);
  const int H = L->hidden, KV = L->kv, I = L->inter;
  const Q82Job jobs[5] = {
      {L->q.codes, L->q.row_scale, L->q.col_field, H, 0, q, PGQ_EPI_NONE, nullptr},
      {L->k.codes, L->k.row_scale, L->k.col_field, KV, 0, k, PGQ_EPI_NONE, nullptr},
      {L->v.codes, L->v.row_scale, L->v.col_field, KV, 0, v, PGQ_EPI_NONE, nullptr},
      {L->o.codes, L->o.row_scale, L->o.col_field, H, 1, o, PGQ_EPI_NONE, nullptr},
      {L->up.codes, L->up.row_scale, L->up.col_field, I, 0, u, PGQ_EPI_RELU2, nullptr},
  };
  const pgq_input ins[2] = {{x, gamma}, {x_o, nullptr}};
  int st = gemv_q82f_multi_impl(jobs, 5, ins, 2, H, 1, eps, (flags & PGQ_WEIGHTS_STABLE) ? 1 : 0, stream);
  if (st) return st;
  // the down launch follows the launch above, which writes no weights
  const Q82Job dj{L->down.codes, L->down.row_scale, L->down.col_field, H, 0, down, PGQ_EPI_NONE, nullptr};
  const pgq_input din{u, nullptr};
  return gemv_q82f_multi_impl(&dj, 1, &din, 1, I, 1, 0.f, 1, stream);
}

// ------------------------------------------------------------------ decode workloads
int pgq_mlp_f16_decode(const float* h, const uint16_t* W_up, const uint16_t* W_down, int hidden, int inter,
                       const float* gamma, float eps, float* u, float* y, void* stream) {
  REQUIRE(h && W_up && W_down && gamma && u && y, PGQ_EINVAL, "mlp_f16_decode: null pointer");
  REQUIRE(!overlaps(u, (size_t)inter * 4, h, (size_t)hidden * 4) && !overlaps(u, (size_t)inter * 4, y, (size_t)hidden * 4),
          PGQ_EINVAL, "mlp_f16_decode: u must not overlap h or y");
  int st = pgq_gemv_f16(W_up, inter, hidden, h, 1, gamma, eps, u, PGQ_EPI_RELU2, nullptr, stream);
  if (st) return st;
  // the down launch follows the up launch, which writes no weights (early weight stream)
  return gemv_f16_impl(W_down, hidden, inter, u, 1, nullptr, 0.f, y, PGQ_EPI_ADD, h, 1, stream);
}

int pgq_q8_decode_layer(const pgq_q8_layer* L, const float* x, const float* x_o, const float* gamma, float eps,
                        float* q, float* k, float* v, float* o, float* u, float* down, void* stream) {
  return pgq_q8_decode_layer_ex(L, x, x_o, gamma, eps, q, k, v, o, u, down, 0, stream);
}

int pgq_q8_decode_layer_ex(const pgq_q8_layer* L, const float* x, const float* x_o, const float* gamma, float eps,
                           float* q, float* k, float* v, float* o, float* u, float* down, int flags, void* stream) {
  REQUIRE(L && x && x_o && gamma && q && k && v && o && u && down, PGQ_EINVAL, "q8_decode_layer: null pointer");
  REQUIRE((flags & ~PGQ_WEIGHTS_STABLE) == 0, PGQ_EINVAL, "q8_decode_layer: unknown flags 0x%x", flags);
  const int H = L->hidden, KV = L->kv, I = L->inter;
  pgq_q8_job jobs[5] = {
      {L->q.codes, L->q.params, H, 0, q, PGQ_EPI_NONE, nullptr},
      {L->k.codes, L->k.params, KV, 0, k, PGQ_EPI_NONE, nullptr},
      {L->v.codes, L->v.params, KV, 0, v, PGQ_EPI_NONE, nullptr},
      {L->o.codes, L->o.params, H, 1, o, PGQ_EPI_NONE, nullptr},
      {L->up.codes, L->up.params, I, 0, u, PGQ_EPI_RELU2, nullptr},
  };
  pgq_input ins[2] = {{x, gamma}, {x_o, nullptr}};
  int st = gemv_q8_multi_impl(jobs, 5, ins, 2, H, 1, eps, (flags & PGQ_WEIGHTS_STABLE) ? 1 : 0, stream);
  if (st) return st;
  // the down launch follows the launch above, which writes no weights: its weight
  // stream may start while that launch finishes
  pgq_q8_job dj{L->down.codes, L->down.params, H, 0, down, PGQ_EPI_NONE, nullptr};
  pgq_input din{u, nullptr};
  return gemv_q8_multi_impl(&dj, 1, &din, 1, I, 1, 0.f, 1, stream);
}

// ------------------------------------------------------------------ fused decode layers
static int check_sync(const void* sync) {
  REQUIRE(sync && aligned16(sync), PGQ_EINVAL, "fused layer: the sync word must be non-null and 16-byte aligned");
  return PGQ_OK;
}

int pgq_q8_decode_layer_fused(const pgq_q8_layer* L, const float* x, const float* x_o, const float* gamma, float eps,
                              float* q, float* k, float* v, float* o, float* u, float* down, int flags, void* sync,
                              void* stream) {
  REQUIRE(L && x && x_o && gamma && q && k && v && o && u && down, PGQ_EINVAL, "q8_decode_layer_fused: null pointer");
  REQUIRE((flags & ~PGQ_WEIGHTS_STABLE) == 0, PGQ_EINVAL, "q8_decode_layer_fused: unknown flags 0x%x", flags);
  if (int st = check_sync(sync)) return st;
  const int H = L->hidden, KV = L->kv, I = L->inter;
  pgq_q8_job jobs[5] = {
      {L->q.codes, L->q.params, H, 0, q, PGQ_EPI_NONE, nullptr},
      {L->k.codes, L->k.params, KV, 0, k, PGQ_EPI_NONE, nullptr},
      {L->v.codes, L->v.params, KV, 0, v, PGQ_EPI_NONE, nullptr},
      {L->o.codes, L->o.params, H, 1, o, PGQ_EPI_NONE, nullptr},
      {L->up.codes, L->up.params, I, 0, u, PGQ_EPI_RELU2, nullptr},
  };
  pgq_input ins[2] = {{x, gamma}, {x_o, nullptr}};
  GvParams A{}, Bp{};
  int st = gemv_q8_multi_impl(jobs, 5, ins, 2, H, 1, eps, (flags & PGQ_WEIGHTS_STABLE) ? 1 : 0, stream, &A);
  if (st) return st;
  pgq_q8_job dj{L->down.codes, L->down.params, H, 0, down, PGQ_EPI_NONE, nullptr};
  pgq_input din{u, nullptr};
  if ((st = gemv_q8_multi_impl(&dj, 1, &din, 1, I, 1, 0.f, 1, stream, &Bp))) return st;
  GET_DEVICE(dev);
  st = launch_gemv_layer(A, Bp, true, static_cast<unsigned*>(sync), dev, as_stream(stream));
  if (st == PGQ_EUNSUPPORTED) return set_error(st, "q8_decode_layer_fused: shapes outside the fused kernel's limits");
  return st;
}

int pgq_mlp_f16_decode_fused(const float* h, const uint16_t* W_up, const uint16_t* W_down, int hidden, int inter,
                             const float* gamma, float eps, float* u, float* y, void* sync, void* stream) {
  REQUIRE(h && W_up && W_down && gamma && u && y, PGQ_EINVAL, "mlp_f16_decode_fused: null pointer");
  REQUIRE(!overlaps(u, (size_t)inter * 4, h, (size_t)hidden * 4) && !overlaps(u, (size_t)inter * 4, y, (size_t)hidden * 4),
          PGQ_EINVAL, "mlp_f16_decode_fused: u must not overlap h or y");
  if (int st = check_sync(sync)) return st;
  GvParams A{}, Bp{};
  int st = gemv_f16_impl(W_up, inter, hidden, h, 1, gamma, eps, u, PGQ_EPI_RELU2, nullptr, 0, stream, &A);
  if (st) return st;
  if ((st = gemv_f16_impl(W_down, hidden, inter, u, 1, nullptr, 0.f, y, PGQ_EPI_ADD, h, 1, stream, &Bp))) return st;
  GET_DEVICE(dev);
  st = launch_gemv_layer(A, Bp, false, static_cast<unsigned*>(sync), dev, as_stream(stream));
  if (st == PGQ_EUNSUPPORTED) return set_error(st, "mlp_f16_decode_fused: shapes outside the fused kernel's limits");
  return st;
}

// ------------------------------------------------------------------ prefill


size_t pgq_prefill_q8_workspace_bytes(const int* rows, int njobs, int cols, int B) {
  if (!rows || njobs < 1 || njobs > TC_MAXJOBS || cols < 128 || B < 1 || B > PGQ_PASS_BMAX) return 0;
  DeviceInfo dev;
  if (!device_info(&dev)) dev.sms = 160;
  return prefill_workspace_bytes(rows, njobs, cols, B, dev);
}

int pgq_prefill_q8(const pgq_q8_job* jobs, int njobs, const float* X, int cols, int B, void* workspace,
                   size_t workspace_bytes, void* stream) {
  REQUIRE(jobs && X, PGQ_EINVAL, "prefill_q8: jobs and X must be non-null");
  REQUIRE(njobs >= 1 && njobs <= TC_MAXJOBS, PGQ_EINVAL, "prefill_q8: njobs=%d outside 1..%d", njobs, TC_MAXJOBS);
  REQUIRE(B >= 1 && B <= PGQ_PASS_BMAX, PGQ_EINVAL, "prefill_q8: B=%d outside 1..%d", B, PGQ_PASS_BMAX);
  REQUIRE(cols >= 128 && cols % 128 == 0, PGQ_EUNSUPPORTED, "prefill_q8: cols=%d must be a multiple of 128", cols);
  REQUIRE(aligned16(X), PGQ_EALIGN, "prefill_q8: X must be 16-byte aligned");
  REQUIRE(workspace && ((uintptr_t)workspace & 255) == 0, PGQ_EWORKSPACE,
          "prefill_q8: workspace must be non-null and 256-byte aligned");
  PrefillJob pj[TC_MAXJOBS];
  int rows[TC_MAXJOBS];
  for (int j = 0; j < njobs; ++j) {
    const pgq_q8_job& J = jobs[j];
    REQUIRE(J.codes && J.params && J.y, PGQ_EINVAL, "prefill_q8: job %d has a null codes/params/y", j);
    REQUIRE(J.rows >= 1, PGQ_EINVAL, "prefill_q8: job %d rows=%d", j, J.rows);
    REQUIRE(aligned16(J.codes) && aligned16(J.params), PGQ_EALIGN, "prefill_q8: job %d codes/params 16-byte", j);
    REQUIRE(aligned4(J.y) && (!J.residual || aligned4(J.residual)), PGQ_EALIGN, "prefill_q8: job %d y/residual", j);
    REQUIRE(J.epilogue >= PGQ_EPI_NONE && J.epilogue <= PGQ_EPI_ADD, PGQ_EINVAL, "prefill_q8: bad epilogue");
    REQUIRE(J.epilogue != PGQ_EPI_ADD || J.residual, PGQ_EINVAL, "prefill_q8: PGQ_EPI_ADD needs a residual");
    const size_t yb = (size_t)B * J.rows * 4;
    REQUIRE(!overlaps(J.y, yb, X, (size_t)B * cols * 4), PGQ_EINVAL, "prefill_q8: job %d output overlaps X", j);
    REQUIRE(!J.residual || J.residual == J.y || !overlaps(J.y, yb, J.residual, yb), PGQ_EINVAL,
            "prefill_q8: residual must be y itself or not overlap it");
    REQUIRE(!overlaps(J.y, yb, workspace, workspace_bytes), PGQ_EINVAL, "prefill_q8: output overlaps workspace");
    pj[j] = PrefillJob{J.codes, J.params, J.rows, J.y, J.residual, J.epilogue};
    rows[j] = J.rows;
  }
  GET_DEVICE(dev);
  const size_t need = prefill_workspace_bytes(rows, njobs, cols, B, dev);
  REQUIRE(workspace_bytes >= need, PGQ_EWORKSPACE, "prefill_q8: workspace needs %zu bytes", need);
  return launch_prefill(pj, njobs, X, cols, B, workspace, workspace_bytes, 0, dev, as_stream(stream));
}

int pgq_prefill_q82f(const pgq_q82f_job* jobs, int njobs, const float* X, int cols, int B, void* workspace,
                     size_t workspace_bytes, void* stream) {
  REQUIRE(jobs && X, PGQ_EINVAL, "prefill_q82f: jobs and X must be non-null");
  REQUIRE(njobs >= 1 && njobs <= TC_MAXJOBS, PGQ_EINVAL, "prefill_q82f: njobs=%d outside 1..%d", njobs, TC_MAXJOBS);
  REQUIRE(B >= 1 && B <= PGQ_PASS_BMAX, PGQ_EINVAL, "prefill_q82f: B=%d outside 1..%d", B, PGQ_PASS_BMAX);
  REQUIRE(cols >= 128 && cols % 128 == 0, PGQ_EUNSUPPORTED, "prefill_q82f: cols=%d must be a multiple of 128", cols);
  REQUIRE(aligned16(X), PGQ_EALIGN, "prefill_q82f: X must be 16-byte aligned");
  REQUIRE(workspace && ((uintptr_t)workspace & 255) == 0, PGQ_EWORKSPACE,
          "prefill_q82f: workspace must be non-null and 256-byte aligned");
  PrefillJob pj[TC_MAXJOBS];
  int rows[TC_MAXJOBS];
  for (int j = 0; j < njobs; ++j) {
    const pgq_q82f_job& J = jobs[j];
    REQUIRE(J.codes && J.row_scale && J.col_field && J.y, PGQ_EINVAL,
            "prefill_q82f: job %d has a null codes/row_scale/col_field/y", j);
    REQUIRE(J.rows >= 1, PGQ_EINVAL, "prefill_q82f: job %d rows=%d", j, J.rows);
    REQUIRE(aligned16(J.codes) && aligned16(J.row_scale) && aligned16(J.col_field), PGQ_EALIGN,
            "prefill_q82f: job %d codes/row_scale/col_field 16-byte", j);
    REQUIRE(aligned4(J.y) && (!J.residual || aligned4(J.residual)), PGQ_EALIGN, "prefill_q82f: job %d y/residual", j);
    REQUIRE(J.epilogue >= PGQ_EPI_NONE && J.epilogue <= PGQ_EPI_ADD, PGQ_EINVAL, "prefill_q82f: bad epilogue");
    REQUIRE(J.epilogue != PGQ_EPI_ADD || J.residual, PGQ_EINVAL, "prefill_q82f: PGQ_EPI_ADD needs a residual");
    const size_t yb = (size_t)B * J.rows * 4;
    REQUIRE(!overlaps(J.y, yb, X, (size_t)B * cols * 4), PGQ_EINVAL, "prefill_q82f: job %d output overlaps X", j);
    REQUIRE(!J.residual || J.residual == J.y || !overlaps(J.y, yb, J.residual, yb), PGQ_EINVAL,
            "prefill_q82f: residual must be y itself or not overlap it");
    REQUIRE(!overlaps(J.y, yb, workspace, workspace_bytes), PGQ_EINVAL, "prefill_q82f: output overlaps workspace");
    PrefillJob w{};
    w.codes = J.codes;
    w.rs = J.row_scale;
    w.cf = J.col_field;
    w.rows = J.rows;
    w.y = J.y;
    w.residual = J.residual;
    w.epilogue = J.epilogue;
    pj[j] = w;
    rows[j] = J.rows;
  }
  GET_DEVICE(dev);
  const size_t need = prefill_workspace_bytes(rows, njobs, cols, B, dev);
  REQUIRE(workspace_bytes >= need, PGQ_EWORKSPACE, "prefill_q82f: workspace needs %zu bytes", need);
  return launch_prefill(pj, njobs, X, cols, B, workspace, workspace_bytes, 0, dev, as_stream(stream));
}

// ------------------------------------------------------------------ prefill pass
namespace {
struct PassLayout {
  size_t off[7];   // n1, q, k, v, h1, n2, u
  size_t gemm;     // prefill workspace
  size_t total;
};
PassLayout pass_layout(int H, int KV, int I, int B, const DeviceInfo& dev) {
  PassLayout L{};
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  // the GEMM part first: its status word is at offset 0 (pgq_prefill_status)
  L.gemm = 0;
  size_t o = up(prefill_pass_gemm_bytes(H, KV, I, B, dev));
  const size_t sz[7] = {(size_t)B * H, (size_t)B * H, (size_t)B * KV, (size_t)B * KV,
                        (size_t)B * H, (size_t)B * H, (size_t)B * I};
  for (int i = 0; i < 7; ++i) {
    L.off[i] = o;
    o = up(o + sz[i] * 4);
  }
  L.total = o;
  return L;
}
}  // namespace

size_t pgq_q8_prefill_pass_workspace_bytes(int hidden, int kv, int inter, int B) {
  if (hidden < 128 || kv < 1 || inter < 128 || B < 1 || B > PGQ_PASS_BMAX) return 0;
  DeviceInfo dev;
  if (!device_info(&dev)) dev.sms = 160;
  return pass_layout(hidden, kv, inter, B, dev).total;
}

int pgq_q8_prefill_pass_layout(int hidden, int kv, int inter, int B, size_t offsets[7]) {
  REQUIRE(offsets && hidden >= 128 && kv >= 1 && inter >= 128 && B >= 1 && B <= PGQ_PASS_BMAX, PGQ_EINVAL,
          "prefill_pass_layout: bad arguments");
  DeviceInfo dev;
  if (!device_info(&dev)) dev.sms = 160;
  const PassLayout L = pass_layout(hidden, kv, inter, B, dev);
  for (int i = 0; i < 7; ++i) offsets[i] = L.off[i];
  return PGQ_OK;
}

extern "C++" {
namespace {
template <class Layer>
int prefill_pass_impl(const char* name, const Layer* layers, int L, float* h, int B, const float* gamma1,
                      const float* gamma2, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(layers && h && gamma1 && gamma2 && workspace, PGQ_EINVAL, "%s: null pointer", name);
  REQUIRE(L >= 1, PGQ_EINVAL, "%s: L=%d", name, L);
  REQUIRE(B >= 1 && B <= PGQ_PASS_BMAX, PGQ_EINVAL, "%s: B=%d outside 1..%d", name, B, PGQ_PASS_BMAX);
  REQUIRE(aligned16(h) && aligned16(gamma1) && aligned16(gamma2), PGQ_EALIGN,
          "%s: h, gamma1 and gamma2 must be 16-byte aligned", name);
  const int H = layers[0].hidden, KV = layers[0].kv, I = layers[0].inter;
  for (int l = 0; l < L; ++l)
    REQUIRE(layers[l].hidden == H && layers[l].kv == KV && layers[l].inter == I, PGQ_EINVAL,
            "%s: layer %d has a different shape", name, l);
  REQUIRE(H % 128 == 0 && I % 128 == 0, PGQ_EUNSUPPORTED, "%s: hidden and inter must be multiples of 128", name);
  REQUIRE(((uintptr_t)workspace & 255) == 0, PGQ_EWORKSPACE, "%s: workspace must be 256-byte aligned", name);
  GET_DEVICE(dev);
  const PassLayout PL = pass_layout(H, KV, I, B, dev);
  REQUIRE(workspace_bytes >= PL.total, PGQ_EWORKSPACE, "%s: workspace needs %zu bytes", name, PL.total);
  REQUIRE(!overlaps(h, (size_t)B * H * 4, workspace, workspace_bytes), PGQ_EINVAL, "%s: h overlaps workspace", name);
  char* w = static_cast<char*>(workspace);
  float* n1 = reinterpret_cast<float*>(w + PL.off[0]);
  float* q = reinterpret_cast<float*>(w + PL.off[1]);
  float* k = reinterpret_cast<float*>(w + PL.off[2]);
  float* v = reinterpret_cast<float*>(w + PL.off[3]);
  float* h1 = reinterpret_cast<float*>(w + PL.off[4]);
  float* n2 = reinterpret_cast<float*>(w + PL.off[5]);
  float* u = reinterpret_cast<float*>(w + PL.off[6]);
  const PassTaps taps{n1, q, k, v, h1, n2, u};
  return launch_prefill_pass(layers, L, h, B, gamma1, gamma2, eps, taps, w + PL.gemm, PL.off[0] - PL.gemm, dev,
                             as_stream(stream));
}
}  // namespace
}  // extern "C++"

int pgq_q8_prefill_pass(const pgq_q8_layer* layers, int L, float* h, int B, const float* gamma1,
                        const float* gamma2, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_pass_impl("prefill_pass", layers, L, h, B, gamma1, gamma2, eps, workspace, workspace_bytes, stream);
}

int pgq_q82f_prefill_pass(const pgq_q82f_layer* layers, int L, float* h, int B, const float* gamma1,
                          const float* gamma2, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  if (layers) {
    for (int l = 0; l < L; ++l) {
      const pgq_q82f_matrix* m[6] = {&layers[l].q, &layers[l].k, &layers[l].v, &layers[l].o, &layers[l].up,
                                     &layers[l].down};
      for (int i = 0; i < 6; ++i) {
        REQUIRE(m[i]->codes && m[i]->row_scale && m[i]->col_field, PGQ_EINVAL,
                "q82f_prefill_pass: layer %d matrix %d has a null pointer", l, i);
        REQUIRE(aligned16(m[i]->codes) && aligned16(m[i]->row_scale) && aligned16(m[i]->col_field), PGQ_EALIGN,
                "q82f_prefill_pass: layer %d matrix %d: codes, row_scale and col_field 16-byte aligned", l, i);
      }
    }
  }
  return prefill_pass_impl("q82f_prefill_pass", layers, L, h, B, gamma1, gamma2, eps, workspace, workspace_bytes,
                           stream);
}

// ------------------------------------------------------------------ MoE
int pgq_moe_router(const float* R, int E, int cols, const float* n, int B, float* logits, void* stream) {
  REQUIRE(R && n && logits, PGQ_EINVAL, "moe_router: null pointer");
  REQUIRE(E >= 1 && B >= 1 && cols >= 4 && cols % 4 == 0, PGQ_EINVAL, "moe_router: bad shape E=%d B=%d cols=%d", E, B,
          cols);
  REQUIRE(aligned16(n) && aligned16(R) && aligned4(logits), PGQ_EALIGN, "moe_router: n and R 16-byte, logits 4-byte");
  REQUIRE(!overlaps(logits, (size_t)B * E * 4, n, (size_t)B * cols * 4), PGQ_EINVAL, "moe_router: logits overlap n");
  GET_DEVICE(dev);
  return launch_router(R, n, B, E, cols, logits, dev, as_stream(stream));
}

int pgq_moe_route_topk(const float* logits, int B, int E, int k, int renorm, int32_t* sel, float* w, void* stream) {
  REQUIRE(logits && sel && w, PGQ_EINVAL, "moe_route_topk: null pointer");
  REQUIRE(B >= 1 && E >= 1 && E <= 256 && k >= 1 && k <= E && k <= 32, PGQ_EINVAL,
          "moe_route_topk: B=%d E=%d k=%d out of range", B, E, k);
  REQUIRE(aligned4(logits) && aligned4(sel) && aligned4(w), PGQ_EALIGN, "moe_route_topk: 4-byte alignment");
  GET_DEVICE(dev);
  return launch_route_topk(logits, B, E, k, renorm, sel, w, as_stream(stream));
}

int pgq_moe_group_gather(const int32_t* sel, int B, int k, int E, int32_t* counts, int32_t* offsets, int32_t* entries,
                         const float* x, int n, int xdiv, float* x_gathered, void* stream) {
  REQUIRE(sel && counts && offsets && entries, PGQ_EINVAL, "moe_group_gather: null pointer");
  REQUIRE(B >= 1 && k >= 1 && E >= 1, PGQ_EINVAL, "moe_group_gather: B=%d k=%d E=%d", B, k, E);
  REQUIRE((size_t)B * k + 2 * (size_t)E + 1 <= 12288, PGQ_EUNSUPPORTED, "moe_group_gather: too many entries/experts");
  REQUIRE(!x_gathered || (x && n >= 1 && xdiv >= 1), PGQ_EINVAL, "moe_group_gather: gather needs x, n, xdiv");
  GET_DEVICE(dev);
  return launch_group(sel, B * k, E, counts, offsets, entries, x, n, xdiv, x_gathered, as_stream(stream));
}

int pgq_moe_experts_q8(const int8_t* codes, const uint16_t* params, int E, int rows, int cols, const int32_t* counts,
                       const int32_t* offsets, const int32_t* entries, int nentries, const float* x, int xdiv, float* y,
                       int epilogue, void* stream) {
  REQUIRE(codes && params && counts && offsets && entries && x && y, PGQ_EINVAL, "moe_experts_q8: null pointer");
  REQUIRE(E >= 1 && rows >= 1 && cols >= 32 && cols % 32 == 0 && nentries >= 1 && xdiv >= 1, PGQ_EINVAL,
          "moe_experts_q8: bad shape");
  REQUIRE(cols <= 6144, PGQ_EUNSUPPORTED, "moe_experts_q8: cols=%d > 6144", cols);
  REQUIRE(epilogue == PGQ_EPI_NONE || epilogue == PGQ_EPI_RELU2, PGQ_EINVAL, "moe_experts_q8: epilogue NONE or RELU2");
  REQUIRE(aligned8(codes) && aligned4(params) && aligned16(x) && aligned4(y), PGQ_EALIGN,
          "moe_experts_q8: codes 8-byte, params 4-byte, x 16-byte, y 4-byte aligned");
  GET_DEVICE(dev);
  MoeBankArgs a{codes, params, E, rows, cols, counts, offsets, entries, nentries, x, xdiv, y, epilogue};
  return launch_moe_bank(a, dev, as_stream(stream));
}

int pgq_moe_combine_rmsnorm(float* h, const float* o, const float* eo, const float* w, int k, const float* gamma,
                            float eps, int B, int n, float* y, float* inv_rms, void* stream) {
  REQUIRE(h && eo && w && gamma && y, PGQ_EINVAL, "moe_combine_rmsnorm: null pointer");
  REQUIRE(B >= 1 && k >= 1 && n >= 4 && n % 4 == 0 && n <= 16384, PGQ_EINVAL, "moe_combine_rmsnorm: bad shape");
  REQUIRE(aligned16(h) && (!o || aligned16(o)) && aligned16(eo) && aligned16(gamma) && aligned16(y), PGQ_EALIGN,
          "moe_combine_rmsnorm: h, o, eo, gamma and y must be 16-byte aligned");
  REQUIRE(!overlaps(y, (size_t)B * n * 4, h, (size_t)B * n * 4), PGQ_EINVAL, "moe_combine_rmsnorm: y overlaps h");
  GET_DEVICE(dev);
  return launch_moe_combine(h, o, eo, w, k, gamma, eps, B, n, y, inv_rms, as_stream(stream));
}

namespace {
struct MoeLayout {
  size_t gemm;    // the tensor-core banks' area, first: its status word at offset 0
  size_t gend;    // end of that area
  size_t off[9];  // n, logits, sel, w, counts, offsets, entries, u, eo
  size_t tick;    // the routing tickets (RouteOut::ticks words)
  size_t total;
};
MoeLayout moe_layout(const pgq_moe_layer& L, int B) {
  MoeLayout M{};
  const size_t nb = (size_t)B * L.k;
  DeviceInfo dev;
  if (!device_info(&dev)) dev.sms = 160;
  const size_t g = std::max(moe_bank_tc_workspace_bytes(L.E, L.inter, L.hidden, (int)nb, dev),
                            moe_bank_tc_workspace_bytes(L.E, L.hidden, L.inter, (int)nb, dev));
  M.gemm = 0;
  size_t o = (g + 255) / 256 * 256;
  M.gend = o;
  const size_t sz[9] = {(size_t)B * L.hidden * 4, (size_t)B * L.E * 4, nb * 4, nb * 4, (size_t)L.E * 4,
                        ((size_t)L.E + 1) * 4, nb * 4, nb * L.inter * 4, nb * L.hidden * 4};
  for (int i = 0; i < 9; ++i) {
    M.off[i] = o;
    o = (o + sz[i] + 255) / 256 * 256;
  }
  M.tick = o;
  o += 256;
  M.total = o;
  return M;
}

// The layer's first two launches: add + RMSNorm of h into n (which also clears the
// routing tickets), then the router, whose tail makes the selection and the
// per-expert lists (RouteOut).
int moe_norm_route(float* h, int B, const float* gamma1, float eps, int hidden, const float* router, int E, int k,
                   int renorm, char* w, const MoeLayout& M, const DeviceInfo& dev, cudaStream_t st) {
  REQUIRE(aligned16(h) && aligned16(gamma1) && aligned16(router), PGQ_EALIGN,
          "moe layer: h, gamma1 and the router must be 16-byte aligned");
  REQUIRE(eps >= 0.f, PGQ_EINVAL, "moe layer: eps must be >= 0");
  REQUIRE(!overlaps(h, (size_t)B * hidden * 4, w, M.total), PGQ_EINVAL, "moe layer: h overlaps the workspace");
  float* n = reinterpret_cast<float*>(w + M.off[0]);
  unsigned* tick = reinterpret_cast<unsigned*>(w + M.tick);
  if (int rc = launch_add_rmsnorm(h, nullptr, gamma1, eps, 0.f, 0, B, hidden, n, nullptr, st, tick, RouteOut::ticks))
    return rc;
  const RouteOut ro{k,
                    renorm,
                    reinterpret_cast<int32_t*>(w + M.off[2]),
                    reinterpret_cast<float*>(w + M.off[3]),
                    reinterpret_cast<int32_t*>(w + M.off[4]),
                    reinterpret_cast<int32_t*>(w + M.off[5]),
                    reinterpret_cast<int32_t*>(w + M.off[6]),
                    tick};
  return launch_router(router, n, B, E, hidden, reinterpret_cast<float*>(w + M.off[1]), dev, st, &ro);
}
bool moe_layer_ok(const pgq_moe_layer* L, int B) {
  return L && L->router && L->up_codes && L->up_params && L->down_codes && L->down_params && L->E >= 1 && L->k >= 1 &&
         L->k <= L->E && L->hidden >= 32 && L->inter >= 32 && B >= 1 && B <= PGQ_PASS_BMAX;
}
}  // namespace

size_t pgq_moe_layer_workspace_bytes(const pgq_moe_layer* layer, int B) {
  if (!moe_layer_ok(layer, B)) return 0;
  return moe_layout(*layer, B).total;
}

int pgq_moe_layer_layout(const pgq_moe_layer* layer, int B, size_t offsets[9]) {
  REQUIRE(offsets && moe_layer_ok(layer, B), PGQ_EINVAL, "moe_layer_layout: bad arguments");
  const MoeLayout M = moe_layout(*layer, B);
  for (int i = 0; i < 9; ++i) offsets[i] = M.off[i];
  return PGQ_OK;
}

int pgq_moe_prefill_layer(const pgq_moe_layer* L, float* h, int B, const float* gamma1, const float* gamma2, float eps,
                          float* y, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(moe_layer_ok(L, B) && h && gamma1 && gamma2 && y && workspace, PGQ_EINVAL, "moe_prefill_layer: bad arguments");
  REQUIRE(((uintptr_t)workspace & 255) == 0, PGQ_EWORKSPACE, "moe_prefill_layer: workspace must be 256-byte aligned");
  const MoeLayout M = moe_layout(*L, B);
  REQUIRE(workspace_bytes >= M.total, PGQ_EWORKSPACE, "moe_prefill_layer: workspace needs %zu bytes", M.total);
  REQUIRE(L->hidden % 32 == 0 && L->inter % 32 == 0, PGQ_EINVAL, "moe_prefill_layer: hidden/inter % 32");
  char* w = static_cast<char*>(workspace);
  float* n = reinterpret_cast<float*>(w + M.off[0]);
  float* wts = reinterpret_cast<float*>(w + M.off[3]);
  int32_t* counts = reinterpret_cast<int32_t*>(w + M.off[4]);
  int32_t* offs = reinterpret_cast<int32_t*>(w + M.off[5]);
  int32_t* ents = reinterpret_cast<int32_t*>(w + M.off[6]);
  float* u = reinterpret_cast<float*>(w + M.off[7]);
  float* eo = reinterpret_cast<float*>(w + M.off[8]);
  int rc;
  GET_DEVICE(dev);
  if ((rc = moe_norm_route(h, B, gamma1, eps, L->hidden, L->router, L->E, L->k, L->renorm, w, M, dev,
                           as_stream(stream))))
    return rc;
  const int nent = B * L->k;
  // each bank on the tensor cores where its shape allows, else the expert GEMV kernel;
  // the first bank resets the banks' status word, the second keeps what it records
  auto bank = [&](const int8_t* codes, const uint16_t* params, int rows, int cols, const float* x, int xdiv, float* yb,
                  int epi, bool first) -> int {
    const MoeBankArgs a{codes, params, L->E, rows, cols, counts, offs, ents, nent, x, xdiv, yb, epi};
    const int r = launch_moe_bank_tc(a, w + M.gemm, M.gend - M.gemm, dev, as_stream(stream), first);
    if (r != PGQ_EUNSUPPORTED) return r;
    return pgq_moe_experts_q8(codes, params, L->E, rows, cols, counts, offs, ents, nent, x, xdiv, yb, epi, stream);
  };
  if ((rc = bank(L->up_codes, L->up_params, L->inter, L->hidden, n, L->k, u, PGQ_EPI_RELU2, true))) return rc;
  if ((rc = bank(L->down_codes, L->down_params, L->hidden, L->inter, u, 1, eo, PGQ_EPI_NONE, false))) return rc;
  return pgq_moe_combine_rmsnorm(h, nullptr, eo, wts, L->k, gamma2, eps, B, L->hidden, y, nullptr, stream);
}

namespace {
pgq_moe_layer dims_of(const pgq_moe_q82f_layer& Q) {
  pgq_moe_layer L{};
  L.router = Q.router;
  L.E = Q.E;
  L.k = Q.k;
  L.hidden = Q.hidden;
  L.inter = Q.inter;
  L.renorm = Q.renorm;
  return L;
}
bool moe_q82f_ok(const pgq_moe_q82f_layer* Q, int B) {
  return Q && Q->router && Q->up_codes && Q->up_row_scale && Q->up_col_field && Q->down_codes &&
         Q->down_row_scale && Q->down_col_field && Q->E >= 1 && Q->k >= 1 && Q->k <= Q->E && Q->hidden >= 32 &&
         Q->inter >= 32 && B >= 1 && B <= PGQ_PASS_BMAX;
}
}  // namespace

size_t pgq_moe_q82f_layer_workspace_bytes(const pgq_moe_q82f_layer* layer, int B) {
  if (!moe_q82f_ok(layer, B)) return 0;
  return moe_layout(dims_of(*layer), B).total;
}
int pgq_moe_q82f_layer_layout(const pgq_moe_q82f_layer* layer, int B, size_t offsets[9]) {
  REQUIRE(offsets && moe_q82f_ok(layer, B), PGQ_EINVAL, "moe_q82f_layer_layout: bad arguments");
  const MoeLayout M = moe_layout(dims_of(*layer), B);
  for (int i = 0; i < 9; ++i) offsets[i] = M.off[i];
  return PGQ_OK;
}

int pgq_moe_q82f_prefill_layer(const pgq_moe_q82f_layer* Q, float* h, int B, const float* gamma1, const float* gamma2,
                               float eps, float* y, void* workspace, size_t workspace_bytes, void* stream) {
  REQUIRE(moe_q82f_ok(Q, B) && h && gamma1 && gamma2 && y && workspace, PGQ_EINVAL,
          "moe_q82f_prefill_layer: bad arguments");
  REQUIRE(((uintptr_t)workspace & 255) == 0, PGQ_EWORKSPACE, "moe_q82f_prefill_layer: workspace must be 256-byte aligned");
  // the banks run on the tensor cores only: what they take is checked before any launch
  REQUIRE(Q->E <= PGQ_MOE_Q82F_EMAX && Q->hidden % 32 == 0 && Q->inter % 32 == 0, PGQ_EUNSUPPORTED,
          "moe_q82f_prefill_layer: E=%d (at most %d), hidden %d and inter %d (multiples of 32)", Q->E,
          PGQ_MOE_Q82F_EMAX, Q->hidden, Q->inter);
  REQUIRE(aligned16(Q->up_codes) && aligned16(Q->up_row_scale) && aligned16(Q->up_col_field) &&
              aligned16(Q->down_codes) && aligned16(Q->down_row_scale) && aligned16(Q->down_col_field),
          PGQ_EALIGN, "moe_q82f_prefill_layer: codes, row scales and column fields 16-byte aligned");
  const pgq_moe_layer D = dims_of(*Q);
  const MoeLayout M = moe_layout(D, B);
  REQUIRE(workspace_bytes >= M.total, PGQ_EWORKSPACE, "moe_q82f_prefill_layer: workspace needs %zu bytes", M.total);
  char* w = static_cast<char*>(workspace);
  float* n = reinterpret_cast<float*>(w + M.off[0]);
  float* wts = reinterpret_cast<float*>(w + M.off[3]);
  int32_t* counts = reinterpret_cast<int32_t*>(w + M.off[4]);
  int32_t* offs = reinterpret_cast<int32_t*>(w + M.off[5]);
  int32_t* ents = reinterpret_cast<int32_t*>(w + M.off[6]);
  float* u = reinterpret_cast<float*>(w + M.off[7]);
  float* eo = reinterpret_cast<float*>(w + M.off[8]);
  int rc;
  GET_DEVICE(dev);
  if ((rc = moe_norm_route(h, B, gamma1, eps, Q->hidden, Q->router, Q->E, Q->k, Q->renorm, w, M, dev,
                           as_stream(stream))))
    return rc;
  const int nent = B * Q->k;
  auto bank = [&](const int8_t* codes, const uint16_t* rs, const uint16_t* cf, int rows, int cols, const float* x,
                  int xdiv, float* yb, int epi, bool first) -> int {
    MoeBankArgs a{codes, nullptr, Q->E, rows, cols, counts, offs, ents, nent, x, xdiv, yb, epi};
    a.rs = rs;
    a.cf = cf;
    return launch_moe_bank_tc(a, w + M.gemm, M.gend - M.gemm, dev, as_stream(stream), first);
  };
  if ((rc = bank(Q->up_codes, Q->up_row_scale, Q->up_col_field, Q->inter, Q->hidden, n, Q->k, u, PGQ_EPI_RELU2,
                 true)))
    return rc;
  if ((rc = bank(Q->down_codes, Q->down_row_scale, Q->down_col_field, Q->hidden, Q->inter, u, 1, eo, PGQ_EPI_NONE,
                 false)))
    return rc;
  return pgq_moe_combine_rmsnorm(h, nullptr, eo, wts, Q->k, gamma2, eps, B, Q->hidden, y, nullptr, stream);
}

int pgq_prefill_status(const void* workspace, void* stream) {
  REQUIRE(workspace, PGQ_EINVAL, "prefill_status: null workspace");
  GET_DEVICE(dev);
  int v[2] = {PGQ_OK, PGQ_OK};   // the status word, then a second one (reserved)
  cudaError_t e = cudaMemcpyAsync(v, static_cast<const char*>(workspace) + prefill_status_offset(), sizeof(v),
                                  cudaMemcpyDeviceToHost, as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_status(e);
  return v[0] != PGQ_OK ? v[0] : v[1];
}

}  // extern "C"
