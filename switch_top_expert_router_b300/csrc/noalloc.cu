// switch_moe_route_from_logits_noalloc: routing on given logits without any
// caller-provided workspace.
//
// Some callers cannot allocate device memory when they route a batch: for
// example a serving process that handed all of its device memory to a pool
// at start-up and forbids cudaMalloc afterwards, or a runtime whose memory
// budget is fixed before any request arrives.  This entry point keeps its
// scratch (per-CTA histograms and probability sums, ranks, per-expert token
// lists, counters) in one file-scope device array instead of a workspace
// argument, so the caller passes only the logits and the outputs.
//
// The array is static device memory: every GPU that loads the library holds
// it until the process exits, and it bounds the sizes this entry point
// accepts (kNoAllocMaxT tokens, kNoAllocMaxN experts).  All calls share it,
// so two calls that overlap on the GPU (different streams, or different
// host threads on the same device) race on it; calls on one stream are
// ordered and safe.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace smoe {
namespace {

constexpr int64_t kNoAllocMaxT = 16384;
constexpr int64_t kNoAllocMaxN = 256;
constexpr int64_t kNoAllocMaxR = (kNoAllocMaxT + kRouterTM - 1) / kRouterTM;

constexpr size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Scratch layout (bytes), every region 256-byte aligned.
constexpr size_t kOffPpart = 0;
constexpr size_t kOffHist = kOffPpart + up256(kNoAllocMaxR * kNoAllocMaxN * 4);
constexpr size_t kOffRank = kOffHist + up256(kNoAllocMaxR * kNoAllocMaxN * 4);
constexpr size_t kOffPsum = kOffRank + up256(kNoAllocMaxT * 4);
constexpr size_t kOffStart = kOffPsum + up256(kNoAllocMaxN * 4);
constexpr size_t kOffList = kOffStart + up256((kNoAllocMaxN + 1) * 4);
constexpr size_t kOffEntries = kOffList + up256(kNoAllocMaxT * 4);
constexpr size_t kOffCtrl = kOffEntries + up256(kNoAllocMaxN * 8);   // one work item per expert
constexpr size_t kScratchBytes = kOffCtrl + 256;                    // about 1.2 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev];   // device address of g_noalloc_scratch, per device

// Set-up, once per device, with that device current: the host-side name of
// the array is only a stand-in, so ask the runtime for its device address.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace
}  // namespace smoe

using namespace smoe;

extern "C" int switch_moe_route_from_logits_noalloc(const switch_moe_params* p,
                                                    const float* logits, int32_t* expert_id,
                                                    float* gate, int32_t* slot,
                                                    uint8_t* drop_mask, int32_t* expert_counts,
                                                    float* aux_loss,
                                                    switch_moe_stream_t stream) {
  if (!p || !expert_counts || !aux_loss) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->N < 1 || !(p->capacity_factor > 0.0) ||
      (p->priority_mode != SWITCH_MOE_TOKEN_ORDER && p->priority_mode != SWITCH_MOE_GATE_PRIORITY))
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->top_k < 0 || p->top_k > 2 || p->renormalize != 0) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->expand > 1 || p->top_k > 1 || p->expert_choice != 0)
    return SWITCH_MOE_ERR_UNSUPPORTED;   // plain top-1 only
  // sizes past the static scratch are refused, never truncated
  if (p->T > kNoAllocMaxT || p->N > kNoAllocMaxN) return SWITCH_MOE_ERR_UNSUPPORTED;
  int* status = device_status_ptr();
  if (!status) return SWITCH_MOE_ERR_NO_DEVICE;
  void* ws = scratch_for_current_device();
  if (!ws) return SWITCH_MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = (int)p->T, N = (int)p->N;
  if (T == 0) {
    if (cudaMemsetAsync(expert_counts, 0, (size_t)N * 4, s) != cudaSuccess ||
        cudaMemsetAsync(aux_loss, 0, 4, s) != cudaSuccess)
      return SWITCH_MOE_ERR_CUDA;
    return SWITCH_MOE_OK;
  }
  const int64_t C = switch_moe_capacity(p->T, p->N, p->capacity_factor);
  if (C < 1) return SWITCH_MOE_ERR_INVALID_ARG;
  if (!logits || !expert_id || !gate || !slot || !drop_mask) return SWITCH_MOE_ERR_INVALID_ARG;
  if (((uintptr_t)logits | (uintptr_t)expert_id | (uintptr_t)gate | (uintptr_t)slot |
       (uintptr_t)expert_counts | (uintptr_t)aux_loss) & 3u)
    return SWITCH_MOE_ERR_ALIGNMENT;
  int32_t* ctrl = at<int32_t>(ws, kOffCtrl);

  // The router zeroes the scan's done counter (ctrl[0]) itself; every other
  // scratch region is fully written before it is read, so nothing left over
  // from an earlier call is ever used.
  RouterArgs ra{};
  ra.logits_in = logits;
  ra.T = T; ra.d = 8; ra.N = N; ra.x_is_bf16 = 0;
  ra.expert_id = expert_id; ra.gate = gate;
  ra.P_part = at<float>(ws, kOffPpart); ra.hist = at<int32_t>(ws, kOffHist);
  ra.local_rank = at<int32_t>(ws, kOffRank); ra.ctrl = ctrl;
  if (launch_router(ra, s) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;

  ScanArgs sa{};
  sa.hist = ra.hist; sa.P_part = ra.P_part; sa.R = (T + kRouterTM - 1) / kRouterTM; sa.N = N;
  sa.T = T; sa.C = (int)C; sa.counts = expert_counts; sa.P_sum = at<float>(ws, kOffPsum);
  sa.expert_start = at<int32_t>(ws, kOffStart); sa.aux_loss = aux_loss;
  sa.entries = at<int2>(ws, kOffEntries);
  sa.BN = (int)C;   // one work item per expert: no GEMM follows, the list only needs room
  sa.ctrl = ctrl;
  if (launch_scan(sa, s) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;

  AssignArgs aa{};
  aa.T = T; aa.N = N; aa.C = (int)C; aa.d = 8; aa.elem_bytes = 4; aa.mode = p->priority_mode;
  aa.expert_id = expert_id; aa.gate = gate; aa.bases = ra.hist; aa.local_rank = ra.local_rank;
  aa.counts = expert_counts; aa.expert_start = sa.expert_start;
  aa.sorted_list = at<int32_t>(ws, kOffList); aa.slot = slot; aa.drop = drop_mask;
  aa.x = nullptr; aa.xbuf = nullptr; aa.status = status;
  if (launch_assign(aa, nullptr, s) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  if (p->priority_mode == SWITCH_MOE_GATE_PRIORITY && launch_gate_select(aa, s) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}
