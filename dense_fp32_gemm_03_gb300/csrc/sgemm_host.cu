// sgemm_host.cu -- C = A * B for matrices in host memory (sgemm_host in
// include/sgemm.h): the copies to and from the device happen inside the call,
// overlapped with the multiply.
//
// B is copied first, whole.  Then A follows in row panels on a copy stream, and
// each panel is multiplied on the caller's stream as soon as its rows have
// landed: C_p = A_p * B, through the library's own sgemm().  The panel's rows
// of C go back on a second copy stream while the next panel is multiplied.  So
// a call costs about the copy of B and of the first A panel, the multiplies,
// and the copy of the last C panel, instead of every copy plus the multiply.
// The product is the one the pages define ("Beyond Kernel 7: Closing the Gap to
// cuBLAS on an H100 FP32 GEMM", "The operation"); splitting it by rows of C
// changes no element's sum.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace gb300 {
namespace {

constexpr int kMaxPanels = 8;
constexpr int64_t kPanelAlign = 128;  // panel rows: whole tile rows of the pipelined kernel

// Device staging of one (device, stream): packed copies of A, B and C with row
// pitches rounded up to 4 floats (16 bytes, as the pipelined kernel reads them
// in place), plus the copy streams and the events that order the pipeline.
struct HostStaging {
  float* buf = nullptr;
  size_t bytes = 0;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t landed[kMaxPanels] = {}, multiplied[kMaxPanels] = {};
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, HostStaging> g_staging;
// Buffers replaced by larger ones: work queued earlier may still use them.
std::vector<std::pair<int, void*>> g_retired;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Rows of A and C per panel: one panel below 2048 rows, else M / 6 but at
// least 512 rows (so at most six panels).  Measured on GB300 with pinned host
// memory (per call, copies included): 4096^3 2943 us copied then multiplied,
// 2926 / 2626 / 2500 / 2443 / 2483 us in 1 / 2 / 4 / 6 / 8 panels; 2048^3 530 us,
// 443 us in 4; 1024^3 128 us, 125 us in one panel and slower in more (every
// panel adds a launch).  SGEMM_HOST_PANELS (1..8) sets the count, for tuning.
int64_t panel_rows(int64_t M) {
  int64_t rows = M < 2048 ? M : (M + 5) / 6;
  if (rows < 512) rows = 512;
  if (const char* v = std::getenv("SGEMM_HOST_PANELS")) {
    char* end = nullptr;
    const long n = std::strtol(v, &end, 10);
    if (end && *end == 0 && n >= 1 && n <= kMaxPanels) rows = (M + n - 1) / n;
  }
  return round_up(rows, kPanelAlign);
}

void destroy_sync_objects(HostStaging& s) {
  for (int p = 0; p < kMaxPanels; ++p) {
    if (s.landed[p]) cudaEventDestroy(s.landed[p]);
    if (s.multiplied[p]) cudaEventDestroy(s.multiplied[p]);
    s.landed[p] = s.multiplied[p] = nullptr;
  }
  if (s.start) cudaEventDestroy(s.start);
  if (s.done) cudaEventDestroy(s.done);
  if (s.in) cudaStreamDestroy(s.in);
  if (s.out) cudaStreamDestroy(s.out);
  s.start = s.done = nullptr;
  s.in = s.out = nullptr;
}

// All or nothing: after a failure nothing is left half-made, and the next
// call tries again.
bool create_sync_objects(HostStaging& s) {
  bool ok = cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&s.start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) == cudaSuccess;
  for (int p = 0; ok && p < kMaxPanels; ++p)
    ok = cudaEventCreateWithFlags(&s.landed[p], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s.multiplied[p], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) destroy_sync_objects(s);
  return ok;
}

// The staging of (dev, stream), holding at least `bytes`; nullptr on failure.
HostStaging* acquire(int dev, cudaStream_t stream, size_t bytes, sgemm_status_t* st) {
  std::lock_guard<std::mutex> lock(g_mu);
  HostStaging& s = g_staging[{dev, stream}];
  if (s.in == nullptr && !create_sync_objects(s)) {
    cudaGetLastError();
    *st = SGEMM_ERR_LAUNCH;
    return nullptr;
  }
  if (s.bytes < bytes) {
    if (s.buf) g_retired.emplace_back(dev, s.buf);
    s.buf = nullptr;
    s.bytes = 0;
    if (cudaMalloc(&s.buf, bytes) != cudaSuccess) {
      cudaGetLastError();
      s.buf = nullptr;
      *st = SGEMM_ERR_ALLOC;
      return nullptr;
    }
    s.bytes = bytes;
  }
  *st = SGEMM_OK;
  return &s;
}

bool overlaps(const float* X, int64_t rows, int64_t cols, int64_t ld, const float* C,
              int64_t M, int64_t N, int64_t ldc) {
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(X);
  const uintptr_t x1 = x0 + uintptr_t(((rows - 1) * ld + cols) * 4);
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(C);
  const uintptr_t c1 = c0 + uintptr_t(((M - 1) * ldc + N) * 4);
  return x0 < c1 && c0 < x1;
}

// A 2-D copy of `rows` rows of `cols` floats between pitched buffers.
bool copy_rows(float* dst, int64_t dst_ld, const float* src, int64_t src_ld, int64_t rows,
               int64_t cols, cudaStream_t s) {
  return cudaMemcpy2DAsync(dst, size_t(dst_ld) * 4, src, size_t(src_ld) * 4, size_t(cols) * 4,
                           size_t(rows), cudaMemcpyDefault, s) == cudaSuccess;
}

}  // namespace

void host_staging_release() {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_staging) {
    HostStaging& s = kv.second;
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    if (s.buf) cudaFree(s.buf);
    destroy_sync_objects(s);
  }
  for (auto& r : g_retired) {
    cudaSetDevice(r.first);
    cudaDeviceSynchronize();
    cudaFree(r.second);
  }
  g_staging.clear();
  g_retired.clear();
  cudaSetDevice(cur);
}

}  // namespace gb300

extern "C" sgemm_status_t sgemm_host(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                     const float* B, int64_t ldb, float* C, int64_t ldc,
                                     cudaStream_t stream) {
  using namespace gb300;
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
  if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL) return SGEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (C == nullptr || ldc < N) return SGEMM_ERR_INVALID_VALUE;
  if (K > 0 && (A == nullptr || B == nullptr || lda < K || ldb < N)) return SGEMM_ERR_INVALID_VALUE;
  if (K > 0 && (overlaps(A, M, K, lda, C, M, N, ldc) || overlaps(B, K, N, ldb, C, M, N, ldc)))
    return SGEMM_ERR_INVALID_VALUE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED;

  const int64_t kp = round_up(K, 4), np = round_up(N, 4);
  const size_t floats = size_t(M) * kp + size_t(K) * np + size_t(M) * np;
  sgemm_status_t st = SGEMM_OK;
  HostStaging* s = acquire(dev, stream, floats * 4, &st);
  if (s == nullptr) return st;
  float* dA = s->buf;
  float* dB = dA + size_t(M) * kp;
  float* dC = dB + size_t(K) * np;

  // Nothing of this call starts before the work already queued on `stream`
  // (which may still use the staging or the host buffers) has finished.
  if (cudaEventRecord(s->start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(s->in, s->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(s->out, s->start, 0) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;

  const int64_t rows = K > 0 ? panel_rows(M) : M;
  const int panels = int((M + rows - 1) / rows);
  if (K > 0 && !copy_rows(dB, np, B, ldb, K, N, s->in)) return SGEMM_ERR_LAUNCH;
  for (int p = 0; p < panels; ++p) {
    const int64_t r0 = int64_t(p) * rows, nr = (M - r0 < rows) ? M - r0 : rows;
    if (K > 0) {
      if (!copy_rows(dA + size_t(r0) * kp, kp, A + size_t(r0) * lda, lda, nr, K, s->in) ||
          cudaEventRecord(s->landed[p], s->in) != cudaSuccess ||
          cudaStreamWaitEvent(stream, s->landed[p], 0) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    }
    // K == 0 zero-fills the panel of C (the empty sum).
    st = sgemm(nr, N, K, dA + size_t(r0) * kp, kp, dB, np, dC + size_t(r0) * np, np, stream);
    if (st != SGEMM_OK) return st;
    if (cudaEventRecord(s->multiplied[p], stream) != cudaSuccess ||
        cudaStreamWaitEvent(s->out, s->multiplied[p], 0) != cudaSuccess ||
        !copy_rows(C + size_t(r0) * ldc, ldc, dC + size_t(r0) * np, np, nr, N, s->out))
      return SGEMM_ERR_LAUNCH;
  }
  // The caller's stream completes only after C is in host memory.
  if (cudaEventRecord(s->done, s->out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, s->done, 0) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  return SGEMM_OK;
}
