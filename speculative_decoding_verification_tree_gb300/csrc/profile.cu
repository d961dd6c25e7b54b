// Optional per-kernel timing: when enabled, every launch of a profiled kernel
// kind (or every n-th, a sample that keeps the events' own cost off most
// launches) is bracketed by a pair of CUDA events recorded on the launching
// stream.  Reading the totals waits for the recorded events.  Not
// thread-safe: meant for a benchmark driving one stream.
#include <vector>

#include "kernels.h"

namespace sv {
namespace {

constexpr int kMaxPairs = 1 << 14;

constexpr int kKinds = 8;

struct Prof {
  bool on = false;
  int period = 1;                 // bracket every period-th launch of a kind
  int seen[kKinds] = {};          // launches of each kind since enabled
  std::vector<cudaEvent_t> ev;    // 2 per pair
  std::vector<int> kind;          // kind of each recorded pair
  int used = 0;
  int open = -1;                  // pair awaiting its end event
  int dropped = 0;
};
Prof g_prof;

}  // namespace

void prof_begin(int kind, cudaStream_t st) {
  Prof& p = g_prof;
  if (!p.on) return;
  if (kind >= 0 && kind < kKinds && p.seen[kind]++ % p.period != 0) return;
  if (p.used >= kMaxPairs) {
    ++p.dropped;
    return;
  }
  if (p.ev.size() < (size_t)2 * (p.used + 1)) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return;
    }
    p.ev.push_back(a);
    p.ev.push_back(b);
    p.kind.push_back(kind);
  }
  p.kind[p.used] = kind;
  cudaEventRecord(p.ev[2 * p.used], st);
  p.open = p.used;
}

void prof_end(int kind, cudaStream_t st) {
  Prof& p = g_prof;
  if (!p.on || p.open < 0 || p.kind[p.open] != kind) return;
  cudaEventRecord(p.ev[2 * p.open + 1], st);
  p.used = p.open + 1;
  p.open = -1;
}

}  // namespace sv

using namespace sv;

extern "C" {

int spec_profile_enable(int on) {
  if (on < 0) return SPEC_ERR_ARG;
  g_prof.on = on != 0;
  g_prof.period = on > 1 ? on : 1;
  for (int k = 0; k < kKinds; ++k) g_prof.seen[k] = 0;
  g_prof.used = 0;
  g_prof.open = -1;
  g_prof.dropped = 0;
  return SPEC_OK;
}

int spec_profile_read(int kind, double* total_ms, int* launches) {
  if (!total_ms || !launches) return SPEC_ERR_ARG;
  double tot = 0.0;
  int n = 0;
  for (int i = 0; i < g_prof.used; ++i) {
    if (g_prof.kind[i] != kind) continue;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return SPEC_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return SPEC_ERR_CUDA;
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *launches = n;
  return g_prof.dropped ? SPEC_ERR_SHAPE : SPEC_OK;
}

}  // extern "C"
