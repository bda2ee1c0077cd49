// C ABI of libswitchmoe.so: argument checks, workspace plan, TMA tensor
// maps and the launch sequence of the layer forward.  Declarations and the
// contract of each entry point are in include/switch_moe.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace smoe {

__device__ int g_status;   // per-device status word, read by switch_moe_sync_status

namespace {

constexpr int kMaxDevices = 64;
// SM count the K-split heuristic plans for (B300).  The workspace size must
// not depend on which device is current, so the plan does not query it.
constexpr int kPlanSMs = 148;

struct DeviceInfo {
  bool probed = false;
  bool ok = false;
  int sms = 0;
  int* status = nullptr;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Current device, checked once: compute capability 10.3 (B300, sm_103a).
const DeviceInfo* current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    d.probed = true;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    void* p = nullptr;
    d.ok = (major == 10 && minor == 3) &&
           cudaGetSymbolAddress(&p, g_status) == cudaSuccess && d.sms > 0;
    d.status = static_cast<int*>(p);
    cudaGetLastError();
  }
  return d.ok ? &d : nullptr;
}

// ----------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// bf16 matrix [rows, cols] row-major, boxes of 64 columns (128 B) x box_rows,
// 128-byte swizzle: the K-major operand layout of the tensor-core GEMM.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTileK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ----------------------------------------------------------- plan
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Plan {
  int64_t T, d, F, N;
  int C, R;
  bool bf16;
  int mode, gm, shared;
  int expand;        // Expanded Drop candidates (1 = plain top-1)
  int topk;          // experts per token: 1, or 2 (top-2 token choice)
  int renorm;        // top-2 gates renormalised over the pair
  bool ec;           // expert-choice routing
  bool multi;        // several slots may add into one y row (top-2, expert choice)
  int elem;          // bytes per x/W element
  int BN, BNs;       // token tiles: routed experts, shared expert
  int max_entries;   // N * ceil(C / BN)
  int ksplit;        // K splits of the second routed GEMM
  bool fused;        // combine in the second routed GEMM's epilogue (tensor path, ksplit 1)
  bool ffn;          // fused and BN <= 128: both routed GEMMs in one launch (ffn_tc_kernel)
  int part_units;    // tail-split partial tiles of the tensor-core GEMMs
  // workspace offsets
  bool tc_router;    // bf16 x and N <= kMaxExpertsTc: tensor-core router
  int rsplit;        // K splits of the tensor-core router (few tokens, long d_model)
  size_t o_rpart;    // its partial logits [rsplit][T][N]
  size_t o_cand, o_candp, o_used;   // Expanded Drop and top-2
  size_t o_hist2, o_rank2, o_cnt2, o_e1, o_g1;   // top-2
  size_t o_probt, o_sgate;                        // expert choice; slot gates
  size_t o_Ppart, o_hist, o_rank, o_Psum, o_start, o_list, o_entries, o_ctrl, o_wsplit, o_xbuf,
      o_H0, o_H1, o_O, o_Hs0, o_Hs1, o_Os, o_tok, o_part, o_splitcnt, total;
  // extra for the host-IO entry point
  size_t o_xin, o_y, o_eid, o_gate, o_slot, o_drop, o_cnt, o_aux, total_hostio;
};

int64_t capacity_of(int64_t T, int64_t N, double cf) {
  if (T < 1 || N < 1 || !(cf > 0.0) || !std::isfinite(cf)) return SWITCH_MOE_ERR_INVALID_ARG;
  const double c = std::ceil(cf * (double)T / (double)N);
  if (!(c >= 1.0) || c > 2147483647.0) return SWITCH_MOE_ERR_INVALID_ARG;
  return (int64_t)c;
}

int choose_ksplit(int64_t tiles, int k_blocks, int sms) {
  // Split the long K of the second GEMM only when there are too few tiles
  // to give every SM at least two.
  int s = 1;
  while (s < 8 && tiles * s < 2 * (int64_t)sms && k_blocks % (2 * s) == 0) s *= 2;
  return s;
}

int make_plan(const switch_moe_params* p, Plan* pl, bool need_gemm) {
  if (!p) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->N < 1 || p->d_model < 1 || p->d_ff < 1) return SWITCH_MOE_ERR_INVALID_ARG;
  if (!(p->capacity_factor > 0.0) || !std::isfinite(p->capacity_factor))
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->priority_mode != SWITCH_MOE_TOKEN_ORDER && p->priority_mode != SWITCH_MOE_GATE_PRIORITY)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if ((p->gate_multiply != 0 && p->gate_multiply != 1) ||
      (p->has_shared != 0 && p->has_shared != 1) ||
      (p->dtype != SWITCH_MOE_F32 && p->dtype != SWITCH_MOE_BF16))
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->expand < 0 || p->expand > kMaxCand) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->N > kMaxExperts) return SWITCH_MOE_ERR_UNSUPPORTED;
  if (p->expand > 1 && (p->priority_mode != SWITCH_MOE_TOKEN_ORDER || p->expand > p->N))
    return SWITCH_MOE_ERR_UNSUPPORTED;
  if (p->top_k < 0 || p->top_k > 2 || (p->renormalize != 0 && p->renormalize != 1))
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->renormalize && p->top_k != 2) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->top_k == 2 && (p->priority_mode != SWITCH_MOE_TOKEN_ORDER || p->expand > 1 || p->N < 2))
    return SWITCH_MOE_ERR_UNSUPPORTED;
  if (p->expert_choice != 0 && p->expert_choice != 1) return SWITCH_MOE_ERR_INVALID_ARG;
  if (p->expert_choice && (p->top_k > 1 || p->expand > 1)) return SWITCH_MOE_ERR_UNSUPPORTED;
  if (need_gemm && (p->d_model < 8 || p->d_ff < 8 || p->d_model % 8 || p->d_ff % 8))
    return SWITCH_MOE_ERR_UNSUPPORTED;
  if (p->T > (int64_t)1 << 30 || p->d_model > (1 << 20) || p->d_ff > (1 << 20))
    return SWITCH_MOE_ERR_UNSUPPORTED;
  Plan& q = *pl;
  std::memset(&q, 0, sizeof(q));
  q.T = p->T; q.d = p->d_model; q.F = p->d_ff; q.N = p->N;
  q.bf16 = p->dtype == SWITCH_MOE_BF16;
  q.elem = q.bf16 ? 2 : 4;
  q.mode = p->priority_mode; q.gm = p->gate_multiply; q.shared = p->has_shared;
  q.expand = p->expand > 1 ? p->expand : 1;
  q.topk = p->top_k == 2 ? 2 : 1;
  q.renorm = p->renormalize;
  q.ec = p->expert_choice == 1;
  q.multi = q.topk == 2 || q.ec;
  if (q.T == 0) return SWITCH_MOE_OK;
  const int64_t C = capacity_of(q.T, q.N, p->capacity_factor);
  if (C < 1) return SWITCH_MOE_ERR_INVALID_ARG;
  if (q.N * C > ((int64_t)1 << 30)) return SWITCH_MOE_ERR_UNSUPPORTED;
  if ((q.mode == SWITCH_MOE_GATE_PRIORITY || q.ec) && (C < q.T ? C : q.T) > kGateSortMax)
    return SWITCH_MOE_ERR_UNSUPPORTED;
  q.C = (int)C;
  q.R = (int)cdiv(q.T, kRouterTM);
  if (q.bf16) {
    q.BN = (int)(cdiv(C, 16) * 16 < 256 ? cdiv(C, 16) * 16 : 256);
    q.BNs = (int)(cdiv(q.T, 16) * 16 < 256 ? cdiv(q.T, 16) * 16 : 256);
  } else {
    q.BN = kSimtTileN;
    q.BNs = kSimtTileN;
  }
  q.max_entries = (int)(q.N * cdiv(C, q.BN));
  q.ksplit = 1;
  if (q.bf16 && need_gemm && q.BN > 128) {
    // token tiles up to 128 run the one-launch FFN, which balances its own
    // last wave (measured on the decode shape: 354 against 368 us with a
    // K-split second GEMM and a separate combine)
    const int k2 = (int)cdiv(q.F, kTileK);
    q.ksplit = choose_ksplit((int64_t)q.max_entries * cdiv(q.d, kTileM), k2, kPlanSMs);
  }
  const int64_t NC = q.N * C;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  q.o_Ppart = take((size_t)q.R * q.N * 4);
  q.o_hist = take((size_t)q.R * q.N * 4);
  q.o_rank = take((size_t)q.T * 4);
  q.o_Psum = take((size_t)q.N * 4);
  q.o_start = take((size_t)(q.N + 1) * 4);
  q.o_list = take((size_t)q.T * 4);
  q.o_entries = take((size_t)q.max_entries * 8);
  q.o_ctrl = take(64);
  if (q.expand > 1 || q.topk == 2) {
    q.o_cand = take((size_t)q.T * kMaxCand * 4);
    q.o_candp = take((size_t)q.T * kMaxCand * 4);
  }
  if (q.expand > 1 || q.multi)
    q.o_used = take((size_t)q.N * 4);   // filled slots per expert (passes, choices, selection)
  if (q.ec) {
    q.o_probt = take((size_t)q.N * q.T * 4);
    q.o_e1 = take((size_t)q.T * 4);   // the router's top-1 outputs (statistics only)
    q.o_g1 = take((size_t)q.T * 4);
  }
  if (q.topk == 2) {
    q.o_hist2 = take((size_t)q.R * q.N * 4);
    q.o_rank2 = take((size_t)q.T * 4);
    q.o_cnt2 = take((size_t)q.N * 4);
    q.o_e1 = take((size_t)q.T * 4);   // the router's top-1 outputs (the user's are [T, 2])
    q.o_g1 = take((size_t)q.T * 4);
  }
  q.tc_router = q.bf16 && q.N <= kMaxExpertsTc;
  // Few tokens (at most 8 router tiles of 128) and a long d_model: one CTA
  // per tile would walk every K block alone, so the K blocks are split over
  // more CTAs (at least 4 blocks each); their sums are added and routed by
  // the FFMA router's kernel.
  q.rsplit = 1;
  if (q.tc_router && q.N <= 128) {
    const int64_t tiles = cdiv(q.T, 128), kbt = cdiv(q.d, kTileK);
    if (tiles <= 8)
      while (q.rsplit < 32 && tiles * q.rsplit * 2 <= kPlanSMs && kbt >= 8 * q.rsplit)
        q.rsplit *= 2;
  }
  if (q.rsplit > 1) q.o_rpart = take((size_t)q.rsplit * q.T * q.N * 4);
  if (q.tc_router) q.o_wsplit = take((size_t)3 * router_tc_n_mma((int)q.N) * q.d * 2);
  if (need_gemm) {
    q.o_xbuf = take((size_t)NC * q.d * q.elem);
    if (q.bf16) {
      q.o_H0 = take((size_t)NC * q.F * 2);
      q.o_H1 = take((size_t)NC * q.F * 2);
    } else {
      q.o_H0 = take((size_t)NC * q.F * 4);
    }
    q.fused = q.bf16 && q.ksplit == 1;
    if (q.fused || q.ec) q.o_tok = take((size_t)NC * 4);
    if (q.multi) q.o_sgate = take((size_t)NC * 4);
    if (!q.fused) {
      q.o_O = take((size_t)q.ksplit * NC * q.d * 4);
    }
    q.ffn = q.fused && q.BN <= 128;
    if (q.bf16) {
      q.part_units = kPlanSMs;
      q.o_part = take((size_t)q.part_units * kTileM * q.BN * 4);
      // tail-split counters, then the fused FFN's per-work-item counters and
      // its unit counter; the scan zeroes them every forward
      q.o_splitcnt = take((size_t)(4 * q.part_units + q.max_entries + 1) * 4);
    }
    if (q.shared) {
      if (q.bf16) {
        q.o_Hs0 = take((size_t)q.T * q.F * 2);
        q.o_Hs1 = take((size_t)q.T * q.F * 2);
      } else {
        q.o_Hs0 = take((size_t)q.T * q.F * 4);
      }
      if (!q.fused) q.o_Os = take((size_t)q.T * q.d * 4);   // fused: the shared expert writes y
    }
  }
  q.total = o;
  q.o_xin = take((size_t)q.T * q.d * q.elem);
  q.o_y = take((size_t)q.T * q.d * 4);
  q.o_eid = take((size_t)q.T * q.topk * 4);
  q.o_gate = take((size_t)q.T * q.topk * 4);
  q.o_slot = take((size_t)q.T * q.topk * 4);
  q.o_drop = take((size_t)q.T * q.topk);
  q.o_cnt = take((size_t)q.N * 4);
  q.o_aux = take(4);
  q.total_hostio = o;
  return SWITCH_MOE_OK;
}

inline bool al(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

// Phase events of switch_moe_set_phase_events (per host thread).
thread_local cudaEvent_t t_phase[SWITCH_MOE_NUM_PHASE_EVENTS];
thread_local bool t_phase_on = false;
inline void mark(int i, cudaStream_t s) {
  if (t_phase_on) cudaEventRecord(t_phase[i], s);
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// bf16 router on the tensor cores: split W_g into three bf16 pieces, then
// logits + softmax/top-1/gate/partials in one kernel.
int launch_tc_router(const Plan& q, const RouterArgs& ra, void* ws, int* status, cudaStream_t s) {
  const int n_mma = router_tc_n_mma((int)q.N);
  __nv_bfloat16* pieces = at<__nv_bfloat16>(ws, q.o_wsplit);
  if (launch_split_wg(ra.W_g, pieces, (int)q.N, (int)q.d, s) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  CUtensorMap tx, tw;
  if (!make_map(&tx, ra.x, (uint64_t)q.T, (uint64_t)q.d, 128) ||
      !make_map(&tw, pieces, (uint64_t)3 * n_mma, (uint64_t)q.d, (uint32_t)n_mma))
    return SWITCH_MOE_ERR_CUDA;
  if (q.rsplit == 1) {
    if (launch_router_tc(ra, tx, tw, status, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
    return SWITCH_MOE_OK;
  }
  // split along K: partial sums on the tensor cores, then the parts added in
  // order (+ bias) and routed (or stored, for switch_moe_router_logits)
  RouterArgs rp{};
  rp.x = ra.x; rp.T = ra.T; rp.d = ra.d; rp.N = ra.N; rp.x_is_bf16 = 1;
  rp.part_out = at<float>(ws, q.o_rpart);
  if (launch_router_tc(rp, tx, tw, status, s, true, q.rsplit) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  RouterArgs rr = ra;
  rr.x = nullptr;
  rr.parts_in = rp.part_out;
  rr.n_parts = q.rsplit;
  if (launch_router(rr, s) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

// Routing: router -> scan -> slot assignment (-> gate ranking -> dispatch).
// x == nullptr routes `logits` instead of computing them.
// y (forward with the fused combine, no shared expert): zero rows of dropped tokens.
int run_routing(const Plan& q, const void* x, const float* W_g, const float* b_g,
                const float* logits, int32_t* expert_id, float* gate, int32_t* slot,
                uint8_t* drop, int32_t* counts, float* aux, void* ws, bool dispatch,
                float* y, int* status, cudaStream_t s) {
  int32_t* ctrl = at<int32_t>(ws, q.o_ctrl);
  RouterArgs ra{};
  ra.x = x; ra.W_g = W_g; ra.b_g = b_g; ra.logits_in = logits; ra.logits_out = nullptr;
  ra.T = (int)q.T; ra.d = (int)q.d; ra.N = (int)q.N; ra.x_is_bf16 = q.bf16;
  ra.expert_id = expert_id; ra.gate = gate;
  ra.P_part = at<float>(ws, q.o_Ppart); ra.hist = at<int32_t>(ws, q.o_hist);
  ra.local_rank = at<int32_t>(ws, q.o_rank); ra.ctrl = ctrl;
  ra.n_cand = q.expand > q.topk ? q.expand : q.topk;
  if (ra.n_cand > 1) {
    ra.cand = at<int32_t>(ws, q.o_cand);
    ra.cand_p = at<float>(ws, q.o_candp);
  }
  if (q.topk == 2) {
    // the router's top-1 expert and gate go to scratch; the slot step
    // writes the [T, 2] outputs from the two candidates
    ra.expert_id = at<int32_t>(ws, q.o_e1);
    ra.gate = at<float>(ws, q.o_g1);
    ra.hist2 = at<int32_t>(ws, q.o_hist2);
    ra.local_rank2 = at<int32_t>(ws, q.o_rank2);
  }
  mark(0, s);
  if (x && q.tc_router) {
    int rc = launch_tc_router(q, ra, ws, status, s);
    if (rc) return rc;
  } else if (launch_router(ra, s) != cudaSuccess) {
    return SWITCH_MOE_ERR_CUDA;
  }
  mark(1, s);

  ScanArgs sa{};
  sa.hist = ra.hist; sa.P_part = ra.P_part; sa.R = q.R; sa.N = (int)q.N; sa.T = (int)q.T;
  sa.C = q.C; sa.counts = counts; sa.P_sum = at<float>(ws, q.o_Psum);
  sa.expert_start = at<int32_t>(ws, q.o_start); sa.aux_loss = aux;
  sa.entries = at<int2>(ws, q.o_entries); sa.BN = q.BN; sa.ctrl = ctrl;
  // token order: the assign kernel finishes the pass over experts (work
  // list, L_aux) in an extra CTA while its other CTAs place the tokens
  sa.defer_finish = q.mode == SWITCH_MOE_TOKEN_ORDER;
  if (dispatch && q.part_units) {
    sa.split_cnt = at<int32_t>(ws, q.o_splitcnt);
    sa.n_split_cnt = 4 * q.part_units + q.max_entries + 1;
  }
  if (q.topk == 2) {
    sa.hist2 = ra.hist2;
    sa.counts2 = at<int32_t>(ws, q.o_cnt2);
    sa.kept_out = at<int32_t>(ws, q.o_used);
  }
  if (launch_scan(sa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  mark(2, s);

  AssignArgs aa{};
  aa.T = (int)q.T; aa.N = (int)q.N; aa.C = q.C; aa.d = (int)q.d; aa.elem_bytes = q.elem;
  aa.mode = q.mode; aa.expert_id = expert_id; aa.gate = gate; aa.bases = ra.hist;
  aa.local_rank = ra.local_rank; aa.counts = counts; aa.expert_start = sa.expert_start;
  aa.sorted_list = at<int32_t>(ws, q.o_list); aa.slot = slot; aa.drop = drop;
  aa.x = dispatch ? x : nullptr; aa.xbuf = dispatch ? at<void>(ws, q.o_xbuf) : nullptr;
  aa.tok_of_slot = (dispatch && q.fused) ? at<int32_t>(ws, q.o_tok) : nullptr;
  aa.y = (dispatch && q.fused && !q.shared) ? y : nullptr;
  aa.status = status;
  if (q.topk == 2) {
    aa.topk = 2; aa.renorm = q.renorm;
    aa.cand = ra.cand; aa.cand_p = ra.cand_p;
    aa.bases2 = ra.hist2; aa.local_rank2 = ra.local_rank2;
    aa.eid_out = expert_id; aa.gate_out = gate;
    aa.slot_gate = aa.tok_of_slot ? at<float>(ws, q.o_sgate) : nullptr;
  }
  // with Expanded Drop the work list waits for the last pass (launch_expand)
  const bool finish_here = sa.defer_finish && q.expand == 1;
  if (launch_assign(aa, finish_here ? &sa : nullptr, s, true) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  if (q.expand > 1) {
    // passes 2..k: the tokens still unplaced try their next candidate; the
    // work list and L_aux follow in the same CTA, then the moved rows' copies
    ExpandArgs ea{};
    ea.T = (int)q.T; ea.N = (int)q.N; ea.C = q.C; ea.d = (int)q.d; ea.elem_bytes = q.elem;
    ea.k = q.expand; ea.cand = ra.cand; ea.cand_p = ra.cand_p; ea.counts = counts;
    ea.open = aa.sorted_list;      // unused by token order
    ea.moved = ra.local_rank;      // read by the top-1 pass only
    ea.n_moved = ctrl + 2;
    ea.used = at<int32_t>(ws, q.o_used);
    ea.expert_id = expert_id; ea.gate = gate; ea.slot = slot; ea.drop = drop;
    ea.tok_of_slot = aa.tok_of_slot; ea.x = aa.x; ea.xbuf = aa.xbuf;
    sa.kept = ea.used;
    if (launch_expand(ea, sa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
    if (ea.xbuf && launch_expand_dispatch(ea, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  }
  if (q.mode == SWITCH_MOE_GATE_PRIORITY) {
    if (launch_gate_select(aa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
    if (dispatch && launch_dispatch(aa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  }
  mark(3, s);
  return SWITCH_MOE_OK;
}

// One tensor-core or SIMT GEMM over routed work items or a dense problem.
// combine (layer 2, routed, fused plan): out0 is y; gate and gate_multiply scale it.
int run_gemm(const Plan& q, const DeviceInfo* dev, bool dense, int layer, const void* A,
             const void* B0, const void* B1, void* out0, void* out1, const int32_t* counts,
             const float* gate, void* ws, cudaStream_t s) {
  GemmArgs g{};
  const int64_t M = layer == 1 ? q.F : q.d;
  const int64_t K = layer == 1 ? q.d : q.F;
  const int64_t rows = dense ? q.T : q.C;
  g.M = (int)M; g.K = (int)K; g.rows_per_expert = (int)rows;
  g.BN = dense ? q.BNs : q.BN;
  g.entries = dense ? nullptr : at<int2>(ws, q.o_entries);
  g.n_entries = dense ? nullptr : at<int32_t>(ws, q.o_ctrl) + 1;
  g.n_entries_dense = dense ? (int)cdiv(q.T, g.BN) : 0;
  g.counts = dense ? nullptr : counts;
  g.cap = q.C;
  g.epi = layer == 1 ? 0 : 1;
  g.out0 = out0; g.out1 = out1;
  g.ldo = (int)M;
  g.status = dev->status;
  if (layer == 2 && !dense && q.fused) {
    g.epi = 2;
    g.tok_of_slot = at<int32_t>(ws, q.o_tok);
    g.gate = gate;
    g.gate_multiply = q.gm;
    // top-2: two choices add into a row (zeroed, or holding the shared
    // expert's output); top-1: the shared expert's output is already in y
    g.y_acc = q.multi ? 2 : q.shared;
    g.slot_gate = q.multi ? at<float>(ws, q.o_sgate) : nullptr;
  }
  if (!dense && q.part_units) {
    g.part = at<float>(ws, q.o_part);
    g.part_units = q.part_units;
    g.split_cnt = at<int32_t>(ws, q.o_splitcnt);
  }
  const int64_t n_ent_max = dense ? g.n_entries_dense : q.max_entries;
  if (q.bf16) {
    g.m_tiles = (int)cdiv(M, kTileM);
    g.ksplit = (layer == 2 && !dense) ? q.ksplit : 1;
    g.k_blocks = (int)(cdiv(K, kTileK) / g.ksplit);
    g.num_b = layer == 1 ? 1 : 2;
    g.split_stride = (size_t)q.N * q.C * q.d;
    g.stages = gemm_tc_max_stages(g.BN, g.num_b);
    g.smem_bytes = gemm_tc_smem_bytes(g.BN, g.num_b, g.stages);
    const int64_t tiles_max = n_ent_max * g.m_tiles * g.ksplit;
    g.grid = (int)(tiles_max < dev->sms ? tiles_max : dev->sms);
    if (g.grid < 1) return SWITCH_MOE_OK;
    const int64_t brows = dense ? q.T : q.N * q.C;
    CUtensorMap ta, tb0, tb1;
    if (!make_map(&ta, A, (uint64_t)((dense ? 1 : q.N) * M), (uint64_t)K, kTileM) ||
        !make_map(&tb0, B0, (uint64_t)brows, (uint64_t)K, (uint32_t)g.BN))
      return SWITCH_MOE_ERR_CUDA;
    if (g.num_b == 2) {
      if (!make_map(&tb1, B1, (uint64_t)brows, (uint64_t)K, (uint32_t)g.BN))
        return SWITCH_MOE_ERR_CUDA;
    } else {
      tb1 = tb0;
    }
    if (launch_gemm_tc(g, ta, tb0, tb1, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  } else {
    g.m_tiles = (int)cdiv(M, 64);
    g.ksplit = 1;
    g.k_blocks = 0;
    g.num_b = 1;
    g.split_stride = (size_t)q.N * q.C * q.d;
    const int64_t tiles_max = n_ent_max * g.m_tiles;
    g.grid = (int)tiles_max;
    if (launch_gemm_simt(g, static_cast<const float*>(A), static_cast<const float*>(B0), s,
                         true) != cudaSuccess)
      return SWITCH_MOE_ERR_CUDA;
  }
  return SWITCH_MOE_OK;
}

// Both routed GEMMs in one persistent launch (ffn_tc_kernel).
int run_ffn(const Plan& q, const DeviceInfo* dev, const void* W1, const void* W2, float* y,
            const int32_t* counts, const float* gate, void* ws, cudaStream_t s) {
  FfnArgs a{};
  a.C = q.C; a.BN = q.BN; a.d = (int)q.d; a.F = (int)q.F;
  a.m1 = (int)cdiv(q.F, kTileM); a.kb1 = (int)cdiv(q.d, kTileK);
  a.m2 = (int)cdiv(q.d, kTileM); a.kb2 = (int)cdiv(q.F, kTileK);
  a.entries = at<int2>(ws, q.o_entries);
  a.n_entries = at<int32_t>(ws, q.o_ctrl) + 1;
  a.counts = counts; a.cap = q.C;
  const int64_t units_max = (int64_t)q.max_entries * (a.m1 + a.m2);
  a.grid = (int)(units_max < dev->sms ? units_max : dev->sms);
  if (a.grid < 1) return SWITCH_MOE_OK;
  // a block's GEMM 1 tiles cover about 1.25 waves of the grid, so a block's
  // GEMM 2 tiles start after its GEMM 1 tiles have finished
  int64_t eb = cdiv((int64_t)a.grid * 5, 4 * (int64_t)a.m1);
  const int64_t eb_min = cdiv(q.max_entries, kFfnMaxBlocks);
  if (eb < eb_min) eb = eb_min;
  if (eb < 1) eb = 1;
  a.eb = (int)eb;
  a.dep = at<int32_t>(ws, q.o_splitcnt) + 4 * q.part_units;
  a.sched = a.dep + q.max_entries;
  a.W1 = W1;
  a.n_experts = (int)q.N;
  a.H0 = at<__nv_bfloat16>(ws, q.o_H0); a.H1 = at<__nv_bfloat16>(ws, q.o_H1);
  a.y = y; a.tok_of_slot = at<int32_t>(ws, q.o_tok); a.gate = gate;
  a.gate_multiply = q.gm;
  a.y_acc = q.multi ? 2 : q.shared;
  a.slot_gate = q.multi ? at<float>(ws, q.o_sgate) : nullptr;
  a.part = at<float>(ws, q.o_part); a.part_units = q.part_units;
  a.split_cnt = at<int32_t>(ws, q.o_splitcnt);
  a.stages = ffn_tc_stages(q.BN);
  a.smem_bytes = ffn_tc_smem_bytes(q.BN, a.stages);
  a.status = dev->status;
  const uint64_t rows = (uint64_t)q.N * q.C;
  CUtensorMap tw1, tx, tw2, th0, th1;
  if (!make_map(&tw1, W1, (uint64_t)q.N * q.F, (uint64_t)q.d, kTileM) ||
      !make_map(&tx, at<void>(ws, q.o_xbuf), rows, (uint64_t)q.d, (uint32_t)q.BN) ||
      !make_map(&tw2, W2, (uint64_t)q.N * q.d, (uint64_t)q.F, kTileM) ||
      !make_map(&th0, a.H0, rows, (uint64_t)q.F, (uint32_t)q.BN) ||
      !make_map(&th1, a.H1, rows, (uint64_t)q.F, (uint32_t)q.BN))
    return SWITCH_MOE_ERR_CUDA;
  if (launch_ffn_tc(a, tw1, tx, tw2, th0, th1, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

// Expert-choice routing: router (+ transposed probabilities) -> scan (top-1
// statistics, zeroed per-token counts) -> per-expert selection and dispatch
// (+ work list in an extra CTA).  x == nullptr routes `logits`.
int run_routing_ec(const Plan& q, const void* x, const float* W_g, const float* b_g,
                   const float* logits, int32_t* chosen_token, float* chosen_gate,
                   int32_t* per_token, int32_t* counts, float* aux, void* ws, bool dispatch,
                   float* y, int* status, cudaStream_t s) {
  int32_t* ctrl = at<int32_t>(ws, q.o_ctrl);
  RouterArgs ra{};
  ra.x = x; ra.W_g = W_g; ra.b_g = b_g; ra.logits_in = logits;
  ra.T = (int)q.T; ra.d = (int)q.d; ra.N = (int)q.N; ra.x_is_bf16 = q.bf16;
  ra.expert_id = at<int32_t>(ws, q.o_e1); ra.gate = at<float>(ws, q.o_g1);
  ra.P_part = at<float>(ws, q.o_Ppart); ra.hist = at<int32_t>(ws, q.o_hist);
  ra.local_rank = at<int32_t>(ws, q.o_rank); ra.ctrl = ctrl;
  ra.n_cand = 1;
  ra.probs_t = at<float>(ws, q.o_probt);
  mark(0, s);
  if (x && q.tc_router) {
    int rc = launch_tc_router(q, ra, ws, status, s);
    if (rc) return rc;
  } else if (launch_router(ra, s) != cudaSuccess) {
    return SWITCH_MOE_ERR_CUDA;
  }
  mark(1, s);
  ScanArgs sa{};
  sa.hist = ra.hist; sa.P_part = ra.P_part; sa.R = q.R; sa.N = (int)q.N; sa.T = (int)q.T;
  sa.C = q.C; sa.counts = counts; sa.P_sum = at<float>(ws, q.o_Psum);
  sa.expert_start = at<int32_t>(ws, q.o_start); sa.aux_loss = aux;
  sa.entries = at<int2>(ws, q.o_entries); sa.BN = q.BN; sa.ctrl = ctrl;
  sa.defer_finish = 1;   // the selection kernel's extra CTA runs finish_experts
  if (dispatch && q.part_units) {
    sa.split_cnt = at<int32_t>(ws, q.o_splitcnt);
    sa.n_split_cnt = 4 * q.part_units + q.max_entries + 1;
  }
  sa.kept_all = (int)(q.C < q.T ? q.C : q.T);
  sa.kept_out = at<int32_t>(ws, q.o_used);
  sa.zero_buf = per_token;
  sa.n_zero = (int)q.T;
  if (launch_scan(sa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  mark(2, s);
  ExpertChoiceArgs ea{};
  ea.T = (int)q.T; ea.N = (int)q.N; ea.C = q.C; ea.d = (int)q.d; ea.elem_bytes = q.elem;
  ea.probs_t = ra.probs_t; ea.chosen_token = chosen_token; ea.chosen_gate = chosen_gate;
  ea.per_token = per_token;
  if (dispatch) {
    ea.tok_of_slot = at<int32_t>(ws, q.o_tok);
    ea.slot_gate = at<float>(ws, q.o_sgate);
    ea.x = x; ea.xbuf = at<void>(ws, q.o_xbuf);
    // every slot of a token adds into y: zero it (unless the shared expert
    // stores its output there first)
    ea.y = (q.fused && q.shared) ? nullptr : y;
  }
  ea.status = status;
  if (launch_expert_select(ea, sa, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  mark(3, s);
  return SWITCH_MOE_OK;
}

// The shared expert, the routed experts' FFN and the combine, after routing.
// kept: filled slots per expert (capped at C by the kernels).
int run_experts(const Plan& q, const DeviceInfo* dev, const void* x, const void* W1,
                const void* W2, const void* W1s, const void* W2s, float* y,
                const int32_t* kept, int32_t* expert_id, float* gate, int32_t* slot, void* ws,
                cudaStream_t s) {
  int rc;
  void* xbuf = at<void>(ws, q.o_xbuf);
  void* H0 = at<void>(ws, q.o_H0);
  void* H1 = q.bf16 ? at<void>(ws, q.o_H1) : nullptr;
  // shared expert first: with the fused combine it writes y, which the
  // routed experts' second GEMM then accumulates into
  float* Os = nullptr;
  if (q.shared) {
    void* Hs0 = at<void>(ws, q.o_Hs0);
    void* Hs1 = q.bf16 ? at<void>(ws, q.o_Hs1) : nullptr;
    Os = q.fused ? y : at<float>(ws, q.o_Os);
    if ((rc = run_gemm(q, dev, true, 1, W1s, x, nullptr, Hs0, Hs1, nullptr, gate, ws, s)))
      return rc;
    if ((rc = run_gemm(q, dev, true, 2, W2s, Hs0, Hs1, Os, nullptr, nullptr, gate, ws, s)))
      return rc;
  }
  mark(4, s);
  if (q.ffn) {
    mark(5, s);   // one launch runs both layers
    if ((rc = run_ffn(q, dev, W1, W2, y, kept, gate, ws, s))) return rc;
    mark(6, s);
    mark(7, s);
    return SWITCH_MOE_OK;
  }
  if ((rc = run_gemm(q, dev, false, 1, W1, xbuf, nullptr, H0, H1, kept, gate, ws, s)))
    return rc;
  mark(5, s);
  if (q.fused) {
    // combine runs in the epilogue of the second routed GEMM
    if ((rc = run_gemm(q, dev, false, 2, W2, H0, H1, y, nullptr, kept, gate, ws, s)))
      return rc;
    mark(6, s);
    mark(7, s);
    return SWITCH_MOE_OK;
  }
  float* O = at<float>(ws, q.o_O);
  if ((rc = run_gemm(q, dev, false, 2, W2, H0, H1, O, nullptr, kept, gate, ws, s))) return rc;
  mark(6, s);
  if (q.ec) {
    SlotCombineArgs sc{};
    sc.T = (int)q.T; sc.N = (int)q.N; sc.C = q.C; sc.d = (int)q.d;
    sc.ksplit = q.bf16 ? q.ksplit : 1;
    sc.kept = (int)(q.C < q.T ? q.C : q.T);
    sc.gate_multiply = q.gm;
    sc.tok_of_slot = at<int32_t>(ws, q.o_tok); sc.slot_gate = at<float>(ws, q.o_sgate);
    sc.O = O; sc.split_stride = (size_t)q.N * q.C * q.d; sc.S = Os; sc.y = y;
    if (launch_combine_slots(sc, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
    mark(7, s);
    return SWITCH_MOE_OK;
  }
  CombineArgs ca{};
  ca.T = (int)q.T; ca.d = (int)q.d; ca.C = q.C;
  ca.ksplit = q.bf16 ? q.ksplit : 1;
  ca.gate_multiply = q.gm; ca.topk = q.topk;
  ca.expert_id = expert_id; ca.gate = gate; ca.slot = slot;
  ca.O = O; ca.split_stride = (size_t)q.N * q.C * q.d; ca.S = Os; ca.y = y;
  if (launch_combine(ca, s, true) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  mark(7, s);
  return SWITCH_MOE_OK;
}

int forward_device(const Plan& q, const DeviceInfo* dev, const void* x, const float* W_g,
                   const float* b_g, const void* W1, const void* W2, const void* W1s,
                   const void* W2s, float* y, int32_t* expert_id, float* gate, int32_t* slot,
                   uint8_t* drop, int32_t* counts, float* aux, void* ws, cudaStream_t s) {
  int rc = run_routing(q, x, W_g, b_g, nullptr, expert_id, gate, slot, drop, counts, aux, ws,
                       true, y, dev->status, s);
  if (rc) return rc;
  // filled slots per expert: min(counts, C), or after Expanded Drop its
  // passes' total, or with top-2 both choices' total
  const int32_t* kept = (q.expand > 1 || q.topk == 2) ? at<int32_t>(ws, q.o_used) : counts;
  return run_experts(q, dev, x, W1, W2, W1s, W2s, y, kept, expert_id, gate, slot, ws, s);
}

int forward_ec_device(const Plan& q, const DeviceInfo* dev, const void* x, const float* W_g,
                      const float* b_g, const void* W1, const void* W2, const void* W1s,
                      const void* W2s, float* y, int32_t* chosen_token, float* chosen_gate,
                      int32_t* per_token, int32_t* counts, float* aux, void* ws,
                      cudaStream_t s) {
  int rc = run_routing_ec(q, x, W_g, b_g, nullptr, chosen_token, chosen_gate, per_token, counts,
                          aux, ws, true, y, dev->status, s);
  if (rc) return rc;
  return run_experts(q, dev, x, W1, W2, W1s, W2s, y, at<int32_t>(ws, q.o_used), nullptr,
                     nullptr, nullptr, ws, s);
}

int empty_batch(int32_t* counts, float* aux, int64_t N, cudaStream_t s) {
  if (cudaMemsetAsync(counts, 0, (size_t)N * 4, s) != cudaSuccess ||
      cudaMemsetAsync(aux, 0, 4, s) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

}  // namespace

int* device_status_ptr() {
  const DeviceInfo* d = current_device();
  return d ? d->status : nullptr;
}

}  // namespace smoe

using namespace smoe;

extern "C" {

int64_t switch_moe_capacity(int64_t T, int64_t N, double capacity_factor) {
  return capacity_of(T, N, capacity_factor);
}

int switch_moe_workspace_bytes(const switch_moe_params* p, size_t* bytes) {
  if (!bytes) return SWITCH_MOE_ERR_INVALID_ARG;
  Plan q;
  const int rc = make_plan(p, &q, true);
  if (rc) return rc;
  *bytes = q.total;
  return SWITCH_MOE_OK;
}

int switch_moe_hostio_workspace_bytes(const switch_moe_params* p, size_t* bytes) {
  if (!bytes) return SWITCH_MOE_ERR_INVALID_ARG;
  Plan q;
  const int rc = make_plan(p, &q, true);
  if (rc) return rc;
  *bytes = q.total_hostio;
  return SWITCH_MOE_OK;
}

int switch_moe_forward(const switch_moe_params* p, const void* x, const float* W_g,
                       const float* b_g, const void* W1, const void* W2, const void* W1s,
                       const void* W2s, float* y, int32_t* expert_id, float* gate, int32_t* slot,
                       uint8_t* drop_mask, int32_t* expert_counts, float* aux_loss,
                       void* workspace, size_t workspace_bytes, switch_moe_stream_t stream) {
  Plan q;
  int rc = make_plan(p, &q, true);
  if (rc) return rc;
  if (q.ec || !expert_counts || !aux_loss) return SWITCH_MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (q.T == 0) return empty_batch(expert_counts, aux_loss, q.N, s);
  if (!x || !W_g || !W1 || !W2 || !y || !expert_id || !gate || !slot || !drop_mask || !workspace)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (q.shared && (!W1s || !W2s)) return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(x, 16) || !al(W_g, 16) || !al(W1, 16) || !al(W2, 16) || !al(y, 16) ||
      !al(workspace, 256) || !al(expert_id, 4) || !al(gate, 4) || !al(slot, 4) ||
      !al(expert_counts, 4) || !al(aux_loss, 4) || (b_g && !al(b_g, 4)) ||
      (q.shared && (!al(W1s, 16) || !al(W2s, 16))))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  return forward_device(q, dev, x, W_g, b_g, W1, W2, W1s, W2s, y, expert_id, gate, slot,
                        drop_mask, expert_counts, aux_loss, workspace, s);
}

int switch_moe_forward_hostio(const switch_moe_params* p, const void* x_host, const float* W_g,
                              const float* b_g, const void* W1, const void* W2, const void* W1s,
                              const void* W2s, float* y_host, int32_t* expert_id_host,
                              float* gate_host, int32_t* slot_host, uint8_t* drop_mask_host,
                              int32_t* expert_counts_host, float* aux_loss_host, void* workspace,
                              size_t workspace_bytes, switch_moe_stream_t stream) {
  Plan q;
  int rc = make_plan(p, &q, true);
  if (rc) return rc;
  if (q.ec) return SWITCH_MOE_ERR_INVALID_ARG;   // switch_moe_forward_expert_choice
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  if (!x_host || !W_g || !W1 || !W2 || !y_host || !expert_id_host || !gate_host || !slot_host ||
      !drop_mask_host || !expert_counts_host || !aux_loss_host || !workspace)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (q.shared && (!W1s || !W2s)) return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(W_g, 16) || !al(W1, 16) || !al(W2, 16) || !al(workspace, 256) ||
      (q.shared && (!al(W1s, 16) || !al(W2s, 16))))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total_hostio) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* d_cnt = at<int32_t>(workspace, q.o_cnt);
  float* d_aux = at<float>(workspace, q.o_aux);
  if (q.T == 0) {
    if ((rc = empty_batch(d_cnt, d_aux, q.N, s))) return rc;
  } else {
    void* d_x = at<void>(workspace, q.o_xin);
    if (cudaMemcpyAsync(d_x, x_host, (size_t)q.T * q.d * q.elem, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return SWITCH_MOE_ERR_CUDA;
    // device copies of the outputs live after the forward's own region
    rc = forward_device(q, dev, d_x, W_g, b_g, W1, W2, W1s, W2s, at<float>(workspace, q.o_y),
                        at<int32_t>(workspace, q.o_eid), at<float>(workspace, q.o_gate),
                        at<int32_t>(workspace, q.o_slot), at<uint8_t>(workspace, q.o_drop), d_cnt,
                        d_aux, workspace, s);
    if (rc) return rc;
    const size_t T = (size_t)q.T, Tk = T * q.topk;
    if (cudaMemcpyAsync(y_host, at<void>(workspace, q.o_y), T * q.d * 4, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(expert_id_host, at<void>(workspace, q.o_eid), Tk * 4,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(gate_host, at<void>(workspace, q.o_gate), Tk * 4, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(slot_host, at<void>(workspace, q.o_slot), Tk * 4, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(drop_mask_host, at<void>(workspace, q.o_drop), Tk, cudaMemcpyDeviceToHost,
                        s) != cudaSuccess)
      return SWITCH_MOE_ERR_CUDA;
  }
  if (cudaMemcpyAsync(expert_counts_host, d_cnt, (size_t)q.N * 4, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(aux_loss_host, d_aux, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

int switch_moe_route_from_logits(const switch_moe_params* p, const float* logits,
                                 int32_t* expert_id, float* gate, int32_t* slot,
                                 uint8_t* drop_mask, int32_t* expert_counts, float* aux_loss,
                                 void* workspace, size_t workspace_bytes,
                                 switch_moe_stream_t stream) {
  if (!p) return SWITCH_MOE_ERR_INVALID_ARG;
  switch_moe_params pr = *p;
  pr.d_model = 8;
  pr.d_ff = 8;
  pr.has_shared = 0;
  Plan q;
  int rc = make_plan(&pr, &q, false);
  if (rc) return rc;
  if (q.ec || !expert_counts || !aux_loss) return SWITCH_MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (q.T == 0) return empty_batch(expert_counts, aux_loss, q.N, s);
  if (!logits || !expert_id || !gate || !slot || !drop_mask || !workspace)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(logits, 4) || !al(workspace, 256) || !al(expert_id, 4) || !al(gate, 4) ||
      !al(slot, 4) || !al(expert_counts, 4) || !al(aux_loss, 4))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool on = t_phase_on;
  t_phase_on = false;   // phase events belong to the forward calls only
  rc = run_routing(q, nullptr, nullptr, nullptr, logits, expert_id, gate, slot, drop_mask,
                   expert_counts, aux_loss, workspace, false, nullptr, dev->status, s);
  t_phase_on = on;
  return rc;
}

int switch_moe_forward_expert_choice(const switch_moe_params* p, const void* x, const float* W_g,
                                     const float* b_g, const void* W1, const void* W2,
                                     const void* W1s, const void* W2s, float* y,
                                     int32_t* chosen_token, float* chosen_gate,
                                     int32_t* experts_per_token, int32_t* expert_counts,
                                     float* aux_loss, void* workspace, size_t workspace_bytes,
                                     switch_moe_stream_t stream) {
  Plan q;
  int rc = make_plan(p, &q, true);
  if (rc) return rc;
  if (!q.ec || !expert_counts || !aux_loss) return SWITCH_MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (q.T == 0) return empty_batch(expert_counts, aux_loss, q.N, s);
  if (!x || !W_g || !W1 || !W2 || !y || !chosen_token || !chosen_gate || !experts_per_token ||
      !workspace)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (q.shared && (!W1s || !W2s)) return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(x, 16) || !al(W_g, 16) || !al(W1, 16) || !al(W2, 16) || !al(y, 16) ||
      !al(workspace, 256) || !al(chosen_token, 4) || !al(chosen_gate, 4) ||
      !al(experts_per_token, 4) || !al(expert_counts, 4) || !al(aux_loss, 4) ||
      (b_g && !al(b_g, 4)) || (q.shared && (!al(W1s, 16) || !al(W2s, 16))))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  return forward_ec_device(q, dev, x, W_g, b_g, W1, W2, W1s, W2s, y, chosen_token, chosen_gate,
                           experts_per_token, expert_counts, aux_loss, workspace, s);
}

int switch_moe_route_expert_choice(const switch_moe_params* p, const float* logits,
                                   int32_t* chosen_token, float* chosen_gate,
                                   int32_t* experts_per_token, int32_t* expert_counts,
                                   float* aux_loss, void* workspace, size_t workspace_bytes,
                                   switch_moe_stream_t stream) {
  if (!p) return SWITCH_MOE_ERR_INVALID_ARG;
  switch_moe_params pr = *p;
  pr.d_model = 8;
  pr.d_ff = 8;
  pr.has_shared = 0;
  Plan q;
  int rc = make_plan(&pr, &q, false);
  if (rc) return rc;
  if (!q.ec || !expert_counts || !aux_loss) return SWITCH_MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (q.T == 0) return empty_batch(expert_counts, aux_loss, q.N, s);
  if (!logits || !chosen_token || !chosen_gate || !experts_per_token || !workspace)
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(logits, 4) || !al(workspace, 256) || !al(chosen_token, 4) || !al(chosen_gate, 4) ||
      !al(experts_per_token, 4) || !al(expert_counts, 4) || !al(aux_loss, 4))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool on = t_phase_on;
  t_phase_on = false;
  rc = run_routing_ec(q, nullptr, nullptr, nullptr, logits, chosen_token, chosen_gate,
                      experts_per_token, expert_counts, aux_loss, workspace, false, nullptr,
                      dev->status, s);
  t_phase_on = on;
  return rc;
}

// ------------------------------------------------------------ backward
namespace {

struct BwdPlan {
  size_t o_Xg, o_dO, o_O, o_dX, o_H, o_dH, o_L, o_dgate, o_tok, o_Hs, o_dHs, o_wgpart, total;
  int wg_parts;   // token chunks of dW_g's reduction over the batch
};

int make_bwd_plan(const switch_moe_params* p, Plan* q, BwdPlan* b) {
  int rc = make_plan(p, q, true);
  if (rc) return rc;
  if (q->expand > 1 || q->topk > 1 || q->ec) return SWITCH_MOE_ERR_UNSUPPORTED;   // top-1 only
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  const size_t NC = (size_t)q->N * (q->T ? q->C : 0);
  b->o_Xg = take(NC * q->d * 4);
  b->o_dO = take(NC * q->d * 4);
  b->o_O = take(NC * q->d * 4);
  b->o_dX = take(NC * q->d * 4);
  b->o_H = take(NC * q->F * 4);
  b->o_dH = take(NC * q->F * 4);
  b->o_L = take((size_t)q->T * q->N * 4);
  b->o_dgate = take((size_t)q->T * 4);
  b->o_tok = take(NC * 4);
  b->o_Hs = q->shared ? take((size_t)q->T * q->F * 4) : 0;
  b->o_dHs = q->shared ? take((size_t)q->T * q->F * 4) : 0;
  // dW_g reduces over all T tokens with only N x d outputs: its token range
  // is cut into chunks of at least 256 (at most 32 chunks), summed in order
  b->wg_parts = (int)std::min<int64_t>(32, std::max<int64_t>(1, q->T / 256));
  b->o_wgpart = take((size_t)b->wg_parts * q->N * q->d * 4);
  b->total = o;
  return SWITCH_MOE_OK;
}

BGemmArgs bg(int M, int N, int K, int batches, float* C, bool acc = false) {
  BGemmArgs g{};
  g.M = M; g.N = N; g.K = K; g.batches = batches; g.C = C; g.accumulate = acc;
  return g;
}

}  // namespace

int switch_moe_backward_workspace_bytes(const switch_moe_params* p, size_t* bytes) {
  if (!bytes) return SWITCH_MOE_ERR_INVALID_ARG;
  Plan q;
  BwdPlan b;
  const int rc = make_bwd_plan(p, &q, &b);
  if (rc) return rc;
  *bytes = b.total;
  return SWITCH_MOE_OK;
}

int switch_moe_backward(const switch_moe_params* p, const void* x, const float* W_g,
                        const float* b_g, const void* W1, const void* W2, const void* W1s,
                        const void* W2s, const int32_t* expert_id, const float* gate,
                        const int32_t* slot, const int32_t* expert_counts, const float* dy,
                        float aux_coef, float* dx, float* dW_g, float* db_g, float* dW1,
                        float* dW2, float* dW1s, float* dW2s, void* workspace,
                        size_t workspace_bytes, switch_moe_stream_t stream) {
  Plan q;
  BwdPlan bp;
  int rc = make_bwd_plan(p, &q, &bp);
  if (rc) return rc;
  if (!std::isfinite(aux_coef)) return SWITCH_MOE_ERR_INVALID_ARG;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = (int)q.T, N = (int)q.N, d = (int)q.d, F = (int)q.F, C = q.C;
  if (!dW_g || !dW1 || !dW2 || (q.shared && (!dW1s || !dW2s))) return SWITCH_MOE_ERR_INVALID_ARG;
  if (T == 0) {   // no tokens: every gradient is zero
    if (cudaMemsetAsync(dW_g, 0, (size_t)N * d * 4, s) != cudaSuccess ||
        (db_g && cudaMemsetAsync(db_g, 0, (size_t)N * 4, s) != cudaSuccess) ||
        cudaMemsetAsync(dW1, 0, (size_t)N * F * d * 4, s) != cudaSuccess ||
        cudaMemsetAsync(dW2, 0, (size_t)N * d * F * 4, s) != cudaSuccess ||
        (q.shared && (cudaMemsetAsync(dW1s, 0, (size_t)F * d * 4, s) != cudaSuccess ||
                      cudaMemsetAsync(dW2s, 0, (size_t)d * F * 4, s) != cudaSuccess)))
      return SWITCH_MOE_ERR_CUDA;
    return SWITCH_MOE_OK;
  }
  if (!x || !W_g || !W1 || !W2 || !expert_id || !gate || !slot || !expert_counts || !dy || !dx ||
      !workspace || (q.shared && (!W1s || !W2s)))
    return SWITCH_MOE_ERR_INVALID_ARG;
  if (!al(x, 16) || !al(W_g, 16) || !al(W1, 16) || !al(W2, 16) || !al(dy, 16) || !al(dx, 16) ||
      !al(workspace, 256) || !al(expert_id, 4) || !al(gate, 4) || !al(slot, 4) ||
      !al(expert_counts, 4) || !al(dW_g, 4) || !al(dW1, 4) || !al(dW2, 4) ||
      (b_g && !al(b_g, 4)) || (db_g && !al(db_g, 4)) ||
      (q.shared && (!al(W1s, 16) || !al(W2s, 16) || !al(dW1s, 4) || !al(dW2s, 4))))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < bp.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool bf = q.bf16;
  void* ws = workspace;
  BwdArgs a{};
  a.T = T; a.N = N; a.C = C; a.d = d; a.gate_multiply = q.gm; a.aux_coef = aux_coef;
  a.expert_id = expert_id; a.slot = slot; a.counts = expert_counts; a.gate = gate; a.dy = dy;
  a.Xg = at<float>(ws, bp.o_Xg); a.dO = at<float>(ws, bp.o_dO); a.O = at<float>(ws, bp.o_O);
  a.dX = at<float>(ws, bp.o_dX); a.dx = dx; a.dgate = at<float>(ws, bp.o_dgate);
  a.L = at<float>(ws, bp.o_L); a.b_g = b_g; a.tok = at<int32_t>(ws, bp.o_tok);
  float* H = at<float>(ws, bp.o_H);
  float* dH = at<float>(ws, bp.o_dH);
  const size_t Cd = (size_t)C * d, CF = (size_t)C * F, Fd = (size_t)F * d;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaMemsetAsync(dx, 0, (size_t)T * d * 4, s)) || !ok(launch_bwd_gather(a, x, bf, s)))
    return SWITCH_MOE_ERR_CUDA;
  // routed experts, per expert e over its kept slots (min(count_e, C) rows)
  BGemmArgs g = bg(C, F, d, N, H);                       // Hpre = Xg W1^T
  g.mcount = expert_counts;
  g.a_b = Cd; g.a_m = d; g.a_k = 1; g.b_b = Fd; g.b_n = d; g.b_k = 1;
  g.c_b = CF; g.c_m = F; g.c_n = 1;
  if (!ok(launch_bgemm(g, a.Xg, false, W1, bf, s)) ||
      !ok(launch_bwd_relu(H, expert_counts, C, F, N, s)))   // H = relu(Hpre)
    return SWITCH_MOE_ERR_CUDA;
  if (q.gm) {
    g = bg(C, d, F, N, a.O);                              // O = H W2^T
    g.mcount = expert_counts;
    g.a_b = CF; g.a_m = F; g.a_k = 1; g.b_b = Fd; g.b_n = F; g.b_k = 1;
    g.c_b = Cd; g.c_m = d; g.c_n = 1;
    if (!ok(launch_bgemm(g, H, false, W2, bf, s))) return SWITCH_MOE_ERR_CUDA;
  }
  g = bg(C, F, d, N, dH);                                 // dH = dO W2
  g.mcount = expert_counts;
  g.a_b = Cd; g.a_m = d; g.a_k = 1; g.b_b = Fd; g.b_n = 1; g.b_k = F;
  g.c_b = CF; g.c_m = F; g.c_n = 1;
  if (!ok(launch_bgemm(g, a.dO, false, W2, bf, s)) ||
      !ok(launch_bwd_mask(dH, H, expert_counts, C, F, N, s)))   // through the ReLU
    return SWITCH_MOE_ERR_CUDA;
  g = bg(C, d, F, N, a.dX);                               // dX = dH W1
  g.mcount = expert_counts;
  g.a_b = CF; g.a_m = F; g.a_k = 1; g.b_b = Fd; g.b_n = 1; g.b_k = d;
  g.c_b = Cd; g.c_m = d; g.c_n = 1;
  if (!ok(launch_bgemm(g, dH, false, W1, bf, s))) return SWITCH_MOE_ERR_CUDA;
  g = bg(d, F, C, N, dW2);                                // dW2 = dO^T H over the slots
  g.kcount = expert_counts;
  g.a_b = Cd; g.a_m = 1; g.a_k = d; g.b_b = CF; g.b_n = 1; g.b_k = F;
  g.c_b = Fd; g.c_m = F; g.c_n = 1;
  if (!ok(launch_bgemm(g, a.dO, false, H, false, s))) return SWITCH_MOE_ERR_CUDA;
  g = bg(F, d, C, N, dW1);                                // dW1 = dH^T Xg over the slots
  g.kcount = expert_counts;
  g.a_b = CF; g.a_m = 1; g.a_k = F; g.b_b = Cd; g.b_n = 1; g.b_k = d;
  g.c_b = Fd; g.c_m = d; g.c_n = 1;
  if (!ok(launch_bgemm(g, dH, false, a.Xg, false, s)) || !ok(launch_bwd_scatter(a, s)))
    return SWITCH_MOE_ERR_CUDA;
  if (q.shared) {   // the shared expert, on every token with gate 1
    float* Hs = at<float>(ws, bp.o_Hs);
    float* dHs = at<float>(ws, bp.o_dHs);
    g = bg(T, F, d, 1, Hs);
    g.a_m = d; g.a_k = 1; g.b_n = d; g.b_k = 1; g.c_m = F; g.c_n = 1;
    if (!ok(launch_bgemm(g, x, bf, W1s, bf, s)) || !ok(launch_bwd_relu(Hs, nullptr, T, F, 1, s)))
      return SWITCH_MOE_ERR_CUDA;
    g = bg(T, F, d, 1, dHs);
    g.a_m = d; g.a_k = 1; g.b_n = 1; g.b_k = F; g.c_m = F; g.c_n = 1;
    if (!ok(launch_bgemm(g, dy, false, W2s, bf, s)) ||
        !ok(launch_bwd_mask(dHs, Hs, nullptr, T, F, 1, s)))
      return SWITCH_MOE_ERR_CUDA;
    g = bg(d, F, T, 1, dW2s);
    g.a_m = 1; g.a_k = d; g.b_n = 1; g.b_k = F; g.c_m = F; g.c_n = 1;
    if (!ok(launch_bgemm(g, dy, false, Hs, false, s))) return SWITCH_MOE_ERR_CUDA;
    g = bg(F, d, T, 1, dW1s);
    g.a_m = 1; g.a_k = F; g.b_n = 1; g.b_k = d; g.c_m = d; g.c_n = 1;
    if (!ok(launch_bgemm(g, dHs, false, x, bf, s))) return SWITCH_MOE_ERR_CUDA;
    g = bg(T, d, F, 1, dx, true);
    g.a_m = F; g.a_k = 1; g.b_n = 1; g.b_k = d; g.c_m = d; g.c_n = 1;
    if (!ok(launch_bgemm(g, dHs, false, W1s, bf, s))) return SWITCH_MOE_ERR_CUDA;
  }
  // router: logits again, then the softmax backward through the gate and L_aux
  g = bg(T, N, d, 1, a.L);
  g.a_m = d; g.a_k = 1; g.b_n = d; g.b_k = 1; g.c_m = N; g.c_n = 1;
  if (!ok(launch_bgemm(g, x, bf, W_g, false, s)) || !ok(launch_bwd_router(a, s)))
    return SWITCH_MOE_ERR_CUDA;
  if (db_g && !ok(launch_bwd_colsum(a.L, db_g, T, N, s))) return SWITCH_MOE_ERR_CUDA;
  {                                                       // dW_g = dl^T x over the tokens
    const int parts = bp.wg_parts, chunk = (T + parts - 1) / parts;
    float* wgp = at<float>(ws, bp.o_wgpart);
    g = bg(N, d, T, parts, wgp);
    g.k_chunk = chunk;
    g.a_b = (size_t)chunk * N; g.a_m = 1; g.a_k = N;
    g.b_b = (size_t)chunk * d; g.b_n = 1; g.b_k = d;
    g.c_b = (size_t)N * d; g.c_m = d; g.c_n = 1;
    if (!ok(launch_bgemm(g, a.L, false, x, bf, s)) ||
        !ok(launch_bwd_sum(wgp, parts, (size_t)N * d, dW_g, s)))
      return SWITCH_MOE_ERR_CUDA;
  }
  g = bg(T, d, N, 1, dx, true);                           // dx += dl W_g
  g.a_m = N; g.a_k = 1; g.b_n = 1; g.b_k = d; g.c_m = d; g.c_n = 1;
  if (!ok(launch_bgemm(g, a.L, false, W_g, false, s))) return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

int switch_moe_router_logits(const switch_moe_params* p, const void* x, const float* W_g,
                             const float* b_g, float* logits, void* workspace,
                             size_t workspace_bytes, switch_moe_stream_t stream) {
  Plan q;
  int rc = make_plan(p, &q, false);
  if (rc) return rc;
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  if (q.T == 0) return SWITCH_MOE_OK;
  if (!x || !W_g || !logits || !workspace) return SWITCH_MOE_ERR_INVALID_ARG;
  if (q.d % 8) return SWITCH_MOE_ERR_UNSUPPORTED;
  if (!al(x, 16) || !al(W_g, 16) || !al(logits, 4) || (b_g && !al(b_g, 4)) ||
      !al(workspace, 256))
    return SWITCH_MOE_ERR_ALIGNMENT;
  if (workspace_bytes < q.total) return SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL;
  RouterArgs ra{};
  ra.x = x; ra.W_g = W_g; ra.b_g = b_g; ra.logits_out = logits;
  ra.T = (int)q.T; ra.d = (int)q.d; ra.N = (int)q.N; ra.x_is_bf16 = q.bf16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (q.tc_router) return launch_tc_router(q, ra, workspace, dev->status, s);
  if (launch_router(ra, s) != cudaSuccess) return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

int switch_moe_sync_status(switch_moe_stream_t stream) {
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  return v;
}

const char* switch_moe_strerror(int code) {
  switch (code) {
    case SWITCH_MOE_OK: return "ok";
    case SWITCH_MOE_ERR_INVALID_ARG: return "invalid argument";
    case SWITCH_MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SWITCH_MOE_ERR_UNSUPPORTED: return "shape outside the supported range";
    case SWITCH_MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case SWITCH_MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case SWITCH_MOE_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status code";
  }
}

int switch_moe_set_phase_events(void* const* events, int n) {
  if (!events) {
    t_phase_on = false;
    return SWITCH_MOE_OK;
  }
  if (n != SWITCH_MOE_NUM_PHASE_EVENTS) return SWITCH_MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return SWITCH_MOE_ERR_INVALID_ARG;
    t_phase[i] = static_cast<cudaEvent_t>(events[i]);
  }
  t_phase_on = true;
  return SWITCH_MOE_OK;
}

int switch_moe_selftest_wait_timeout(uint64_t timeout_ns, switch_moe_stream_t stream) {
  const DeviceInfo* dev = current_device();
  if (!dev) return SWITCH_MOE_ERR_NO_DEVICE;
  unsigned long long t = timeout_ns;
  if (t < 1000000ull) t = 1000000ull;
  if (t > 2000000000ull) t = 2000000000ull;
  if (launch_selftest_wait(dev->status, t, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SWITCH_MOE_ERR_CUDA;
  return SWITCH_MOE_OK;
}

int switch_moe_version(void) { return 100; }

}  // extern "C"
