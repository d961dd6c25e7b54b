// spec_verify_chain_noalloc: chain verification for callers that cannot
// allocate device memory.
//
// Who needs it: code that is handed only its input and output buffers and no
// way to get more device memory -- for example an operator plugin inside an
// inference engine that has already carved up all of the GPU's memory, or a
// latency-critical decode loop whose owner forbids cudaMalloc there (it may
// synchronise the device and it can fail at run time).  Such a caller cannot
// provide the workspace spec_verify_chain asks for.
//
// What it does instead: the scratch the verification kernels need (status
// word, per-row outcomes and records, argmax and acceptance-mass partials)
// lives in one file-scope __device__ array of fixed size, which every GPU
// that loads this library holds until the process exits.  Nothing is
// allocated per call.
//
// Rules for callers:
//  * The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
//  * Every call on a device shares the one array and leaves the last call's
//    contents in it; the status word is cleared at the start of each call
//    and read back with spec_get_status_noalloc after it.
//    Calls whose work overlaps on the GPU (other streams, other host threads
//    on the same device) race on the array and must be serialised by the
//    caller.
//  * Sizes: B * (K + 1) <= SPEC_NOALLOC_MAX_ROWS rows and
//    B * (K + 1) * ceil(V / 16384) <= SPEC_NOALLOC_MAX_PARTS argmax partials;
//    larger requests are rejected with SPEC_ERR_SHAPE before any GPU work.
//  * Not served (SPEC_ERR_UNSUPPORTED): sampling with top-k / top-p
//    truncation (its candidate lists need scratch beyond the array), and
//    rows the streaming kernels cannot take (see sampled_supported).  Given
//    draft normalisers (draft_lse) are rejected with SPEC_ERR_ARG.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace sv {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kRowBytes = (size_t)SPEC_NOALLOC_MAX_ROWS * sizeof(int32_t);
constexpr size_t kPartBytes = (size_t)SPEC_NOALLOC_MAX_PARTS * sizeof(ArgPart);
constexpr size_t kAlphaBytes = (size_t)SPEC_NOALLOC_MAX_ROWS * kAlphaSlots * sizeof(float);
constexpr size_t kMetaBytes = (size_t)SPEC_NOALLOC_MAX_ROWS * 48;  // chain row records
constexpr size_t kOutBytes = (size_t)SPEC_NOALLOC_MAX_ROWS * sizeof(RowOut);
constexpr size_t kScratchBytes =
    kStatusBytes + 4 * kRowBytes + kPartBytes + kAlphaBytes + kMetaBytes + kOutBytes;

// The scratch itself (~1.75 MiB per device).  In host code this name is only
// a stand-in; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch for the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return SPEC_OK;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" int spec_verify_chain_noalloc(const void* target_logits, const void* draft,
                                         const int32_t* draft_tokens, int B, int K, int V,
                                         int dtype_target, int dtype_draft,
                                         const spec_params_t* prm, int32_t* accepted,
                                         int32_t* out_tokens, float* accept_mass,
                                         void* stream) {
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_SHAPE;
  if (V > SPEC_MAX_VOCAB || K > SPEC_MAX_TREE_NODES) return SPEC_ERR_SHAPE;
  const int64_t rows = (int64_t)B * (K + 1);
  if (rows > SPEC_NOALLOC_MAX_ROWS) return SPEC_ERR_SHAPE;
  if (rows * arg_splits(V) > SPEC_NOALLOC_MAX_PARTS) return SPEC_ERR_SHAPE;
  if (!prm) return SPEC_ERR_ARG;
  if (!(prm->temperature >= 0.f) || !std::isfinite(prm->temperature)) return SPEC_ERR_ARG;
  if (prm->flags != 0 || prm->top_k < 0 || prm->draft_lse) return SPEC_ERR_ARG;
  if (prm->draft_kind != SPEC_DRAFT_LOGITS && prm->draft_kind != SPEC_DRAFT_PROBS)
    return SPEC_ERR_DTYPE;
  if (!(prm->top_p > 0.f && prm->top_p <= 1.f)) return SPEC_ERR_ARG;
  if (prm->temperature > 0.f && (prm->top_k != 0 || prm->top_p < 1.f)) return SPEC_ERR_UNSUPPORTED;
  if (dtype_target != SPEC_F32 && dtype_target != SPEC_BF16) return SPEC_ERR_DTYPE;
  const bool greedy = prm->temperature == 0.f;
  const bool dt_ok = dtype_draft == SPEC_F32 || dtype_draft == SPEC_BF16;
  if (!greedy && K > 0 && !dt_ok) return SPEC_ERR_DTYPE;
  if (B > 0) {
    if (!target_logits || !accepted || !out_tokens) return SPEC_ERR_ARG;
    if (K > 0 && (!draft_tokens || !accept_mass)) return SPEC_ERR_ARG;
    if (!greedy && K > 0 && !draft) return SPEC_ERR_ARG;
  }
  VerifyShape s{B, K, K, V, true};
  VerifyArgs a{};
  a.target = target_logits;
  a.draft = greedy ? nullptr : draft;
  a.node_tokens = draft_tokens;
  a.dt_target = dtype_target;
  a.dt_draft = dt_ok ? dtype_draft : SPEC_F32;
  a.prm = *prm;
  a.count = accepted;
  a.out_tokens = out_tokens;
  a.mass = accept_mass;
  // the same refusal as the workspace entry point, before the status word
  // of the previous call is cleared
  if (!greedy && !sampled_supported(s, a)) return SPEC_ERR_UNSUPPORTED;
  void* base = nullptr;
  int rc = scratch_address(&base);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  char* p = (char*)base;
  a.status = (uint32_t*)p;
  a.row_child = (int32_t*)(p + kStatusBytes);
  a.row_token = (int32_t*)(p + kStatusBytes + kRowBytes);
  a.arg_part = (ArgPart*)(p + kStatusBytes + 2 * kRowBytes);
  a.alpha_part = (float*)(p + kStatusBytes + 2 * kRowBytes + kPartBytes);
  a.meta = (unsigned char*)(p + kStatusBytes + 2 * kRowBytes + kPartBytes + kAlphaBytes);
  a.qres = (int32_t*)(p + kStatusBytes + 2 * kRowBytes + kPartBytes + kAlphaBytes + kMetaBytes);
  a.rowout = (RowOut*)(p + kStatusBytes + 3 * kRowBytes + kPartBytes + kAlphaBytes + kMetaBytes);
  a.qlist = (int32_t*)(p + kStatusBytes + 3 * kRowBytes + kPartBytes + kAlphaBytes + kMetaBytes +
                       kOutBytes);
  a.qcount = (int32_t*)(p + 4);  // beside the status word, zeroed with it
  if (meta_rec_bytes(true) != 48) return SPEC_ERR_CUDA;  // chain row record size
  // the status word must start at zero (a single-cluster chain launch writes
  // the whole word itself); everything else is written before it is read
  // within the call
  if (!(!greedy && chain_small_writes_status(s, a)) &&
      cudaMemsetAsync(a.status, 0, 2 * sizeof(uint32_t), st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
  const cudaError_t e = greedy ? launch_greedy(s, a, st) : launch_sampled(s, a, st);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_get_status_noalloc(uint32_t* status, void* stream) {
  if (!status) return SPEC_ERR_ARG;
  void* base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // the status word is the first word of the array
  if (cudaMemcpyAsync(status, base, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
