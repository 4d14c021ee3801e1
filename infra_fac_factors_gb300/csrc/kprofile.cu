// Per-launch timing of the main kernels (kfac_profile / kfac_profile_read):
// a record of (kind, start event, end event, work) per launch while
// recording is on.  Events come from a pool that is kept for reuse.
#include <mutex>
#include <vector>

#include "launch.h"

namespace kfac {
namespace {

constexpr size_t kProfCap = 65536;

struct ProfRec {
  int kind;
  cudaEvent_t start, end;
  double work;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_pool;  // events not in use

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void recycle_all() {
  for (const ProfRec& r : g_prof) {
    if (r.start) g_pool.push_back(r.start);
    if (r.end) g_pool.push_back(r.end);
  }
  g_prof.clear();
}

}  // namespace

bool prof_recording() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  return g_prof_on;
}

void prof_begin(cudaStream_t stream, ProfMark& m) {
  m.start = nullptr;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || g_prof.size() >= kProfCap) return;
  m.start = take_event();
  if (m.start && cudaEventRecord(m.start, stream) != cudaSuccess) {
    g_pool.push_back(m.start);
    m.start = nullptr;
  }
}

void prof_end(int kind, cudaStream_t stream, const ProfMark& m, double work) {
  if (!m.start) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t e = take_event();
  if (!e || cudaEventRecord(e, stream) != cudaSuccess) {
    g_pool.push_back(m.start);
    if (e) g_pool.push_back(e);
    return;
  }
  g_prof.push_back(ProfRec{kind, m.start, e, work});
}

}  // namespace kfac

extern "C" {

int kfac_profile(int enable) {
  std::lock_guard<std::mutex> lk(kfac::g_prof_mu);
  if (enable) {
    // the previous record's events may still be pending: wait for them first
    for (const kfac::ProfRec& r : kfac::g_prof) cudaEventSynchronize(r.end);
    kfac::recycle_all();
  }
  kfac::g_prof_on = enable != 0;
  return KFAC_OK;
}

int kfac_profile_read(int kind, int64_t* launches, double* ms, double* work) {
  if (kind < 0 || kind >= KFAC_K_COUNT || !launches || !ms || !work) return KFAC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(kfac::g_prof_mu);
  int64_t n = 0;
  double t = 0.0, w = 0.0;
  for (const kfac::ProfRec& r : kfac::g_prof) {
    if (r.kind != kind) continue;
    if (cudaEventSynchronize(r.end) != cudaSuccess) return KFAC_ERR_CUDA;
    float e = 0.f;
    if (cudaEventElapsedTime(&e, r.start, r.end) != cudaSuccess) return KFAC_ERR_CUDA;
    ++n;
    t += e;
    w += r.work;
  }
  *launches = n;
  *ms = t;
  *work = w;
  return KFAC_OK;
}

int kfac_profile_count(int64_t* count) {
  if (!count) return KFAC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(kfac::g_prof_mu);
  for (const kfac::ProfRec& r : kfac::g_prof)
    if (cudaEventSynchronize(r.end) != cudaSuccess) return KFAC_ERR_CUDA;
  *count = (int64_t)kfac::g_prof.size();
  return KFAC_OK;
}

int kfac_profile_launch(int64_t i, int* kind, double* start_ms, double* end_ms, double* work) {
  if (!kind || !start_ms || !end_ms || !work) return KFAC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(kfac::g_prof_mu);
  if (i < 0 || i >= (int64_t)kfac::g_prof.size()) return KFAC_ERR_INVALID_ARG;
  const kfac::ProfRec& first = kfac::g_prof[0];
  const kfac::ProfRec& r = kfac::g_prof[(size_t)i];
  if (cudaEventSynchronize(r.end) != cudaSuccess || cudaEventSynchronize(first.start) != cudaSuccess)
    return KFAC_ERR_CUDA;
  float a = 0.f, b = 0.f;
  if (cudaEventElapsedTime(&a, first.start, r.start) != cudaSuccess ||
      cudaEventElapsedTime(&b, first.start, r.end) != cudaSuccess)
    return KFAC_ERR_CUDA;
  *kind = r.kind;
  *start_ms = a;
  *end_ms = b;
  *work = r.work;
  return KFAC_OK;
}

}  // extern "C"
