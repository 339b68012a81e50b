// Status strings, the per-device error word and the bounded-wait self test.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace poetx {

// Site id of this file's bounded waits (file id x 10000 + source line), recorded with
// the first timeout.
constexpr int kSite = 4 * 10000;

// Two error words per device (the first error status, the site of the first expired wait);
// kernels receive their address as a parameter and record with atomic compare-and-swaps.
static __device__ int g_error_word[2];

static std::mutex g_mu;
static std::atomic<int*> g_err_ptr[64];
static std::atomic<int> g_sms[64];
static std::atomic<int> g_last_site{0};

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  return dev;
}

int* device_error_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  int* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lk(g_mu);
  p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* v = nullptr;
    if (cudaGetSymbolAddress(&v, g_error_word) != cudaSuccess) return nullptr;
    p = static_cast<int*>(v);
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 148;
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v) return v;
  cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (v <= 0) v = 148;
  g_sms[dev].store(v, std::memory_order_relaxed);
  return v;
}

static std::atomic<unsigned long long> g_launches{0};
static std::atomic<int> g_prof_on{0};
static std::mutex g_prof_mu;
struct ProfRec {
  int stage;  // -1: reference mark
  cudaEvent_t ev;
};
static std::vector<ProfRec> g_prof;
static std::vector<cudaEvent_t> g_prof_pool;

static void prof_record(cudaStream_t s, int stage) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t ev = nullptr;
  if (!g_prof_pool.empty()) {
    ev = g_prof_pool.back();
    g_prof_pool.pop_back();
  } else if (cudaEventCreate(&ev) != cudaSuccess) {
    return;
  }
  cudaEventRecord(ev, s);
  g_prof.push_back({stage, ev});
}

void after_launch(cudaStream_t s, int stage) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof_on.load(std::memory_order_relaxed)) prof_record(s, stage);
}

bool prof_enabled() { return g_prof_on.load(std::memory_order_relaxed); }

void prof_begin(cudaStream_t s) {
  if (g_prof_on.load(std::memory_order_relaxed)) prof_record(s, -1);
}

static const char* kStageNames[ST_COUNT] = {
    "triu_unpack", "cnp_q2", "cnp_g", "cnp_sum_partials", "cnp_m1", "cnp_qbar", "triu_grad_pack",
    "perm_gather", "perm_scatter", "blockdiag_mm", "wprime_gemm", "blockdiag_wgrad",
    "quantize_rows_int8", "merge_perm", "merge_reinit", "adam_triu", "wprime_blockdiag_fused",
    "blockdiag_bwd_fused"};

// Waits on a shared-memory barrier that nothing arrives on, for at most limit_ns, then
// records the timeout and returns.
__global__ void selftest_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, err, limit_ns, kSite + __LINE__);
  __syncthreads();
}

}  // namespace poetx

using namespace poetx;

extern "C" const char* poetx_status_str(poetx_status st) {
  switch (st) {
    case POETX_OK: return "POETX_OK";
    case POETX_ERR_ARG: return "POETX_ERR_ARG: invalid argument";
    case POETX_ERR_SHAPE: return "POETX_ERR_SHAPE: unsupported or inconsistent shape";
    case POETX_ERR_DTYPE: return "POETX_ERR_DTYPE: unsupported dtype";
    case POETX_ERR_ALIGN: return "POETX_ERR_ALIGN: pointer not 16-byte aligned";
    case POETX_ERR_WORKSPACE: return "POETX_ERR_WORKSPACE: workspace too small";
    case POETX_ERR_UNSUPPORTED: return "POETX_ERR_UNSUPPORTED: unsupported option";
    case POETX_ERR_TIMEOUT: return "POETX_ERR_TIMEOUT: a bounded device wait expired";
    case POETX_ERR_CUDA: return "POETX_ERR_CUDA: CUDA runtime error";
  }
  return "POETX_UNKNOWN_STATUS";
}

extern "C" poetx_status poetx_get_device_error(cudaStream_t stream) {
  int* w = device_error_word();
  if (!w) return POETX_ERR_CUDA;
  int host[2] = {0, 0};
  POETX_CUDA_TRY(cudaStreamSynchronize(stream));
  POETX_CUDA_TRY(cudaMemcpy(host, w, sizeof(host), cudaMemcpyDeviceToHost));
  if (host[0] != 0 || host[1] != 0) {
    const int zero[2] = {0, 0};
    POETX_CUDA_TRY(cudaMemcpy(w, zero, sizeof(zero), cudaMemcpyHostToDevice));
    g_last_site.store(host[1]);
  }
  return static_cast<poetx_status>(host[0]);
}

extern "C" poetx_status poetx_selftest_timeout(unsigned int timeout_us, cudaStream_t stream) {
  int* w = device_error_word();
  if (!w) return POETX_ERR_CUDA;
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(w, 1000ull * timeout_us);
  POETX_CUDA_TRY(cudaGetLastError());
  return POETX_OK;
}

extern "C" int poetx_timeout_site(void) { return g_last_site.load(); }

extern "C" unsigned long long poetx_launch_count(void) { return g_launches.load(); }

extern "C" poetx_status poetx_profile_enable(int on) {
  g_prof_on.store(on ? 1 : 0);
  return POETX_OK;
}

extern "C" const char* poetx_stage_name(int stage) {
  return (stage >= 0 && stage < ST_COUNT) ? kStageNames[stage] : "unknown";
}

extern "C" int poetx_profile_collect(int* stage, float* ms, int cap) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int n = 0;
  cudaEvent_t prev = nullptr;
  for (const ProfRec& r : g_prof) {
    cudaEventSynchronize(r.ev);
    if (r.stage >= 0 && prev && n < cap) {
      float t = 0.f;
      cudaEventElapsedTime(&t, prev, r.ev);
      if (stage) stage[n] = r.stage;
      if (ms) ms[n] = t;
      ++n;
    }
    prev = r.ev;
  }
  for (const ProfRec& r : g_prof) g_prof_pool.push_back(r.ev);
  g_prof.clear();
  return n;
}

static std::atomic<unsigned long long*> g_trace{nullptr};
static std::atomic<size_t> g_trace_slots{0};
static std::atomic<size_t> g_trace_next{0};  // region of the next launch

// Each launch gets its own region of kTraceRegionCtas CTAs (the k-th launch since the buffer
// was set writes region k), so that the launches of a captured graph keep separate stamps.
unsigned long long* poetx::trace_buffer(size_t* slots) {
  unsigned long long* base = g_trace.load();
  const size_t total = g_trace_slots.load();
  constexpr size_t region = (size_t)kTraceRegionCtas * kTraceSlots;
  if (!base) {
    *slots = 0;
    return nullptr;
  }
  const size_t k = g_trace_next.fetch_add(1);
  if ((k + 1) * region > total) {
    *slots = 0;
    return nullptr;
  }
  *slots = region;
  return base + k * region;
}

extern "C" poetx_status poetx_set_trace_buffer(void* buf, size_t bytes) {
  if (buf && !aligned16(buf)) return POETX_ERR_ALIGN;
  g_trace_slots.store(buf ? bytes / 8 : 0);
  g_trace_next.store(0);
  g_trace.store(static_cast<unsigned long long*>(buf));
  return POETX_OK;
}
