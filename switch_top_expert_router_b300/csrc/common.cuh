// Internal declarations shared by the library's translation units: kernel
// argument structs and host-side launchers.  Nothing here is exported.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "switch_moe.h"

namespace smoe {

// Launch `k` on `s`; with pdl, as a programmatic dependent launch (the
// kernel may start before the previous kernel of the stream ends and calls
// grid_dep_wait() before it reads that kernel's results).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

constexpr int kRouterTM = 32;        // tokens per router CTA
constexpr int kMaxExperts = 1024;
constexpr int kGateSortMax = 16384;  // keys one gate-priority CTA sorts in shared memory
constexpr int kTileM = 128;          // weight rows per tensor-core tile (MMA M)
constexpr int kTileK = 64;           // bf16 elements per 128-byte K block
constexpr int kSimtTileN = 32;       // tokens per fp32 SIMT tile
constexpr int kMaxExpertsTc = 256;   // experts the tensor-core router takes (one MMA N)
constexpr int kMaxCand = 4;          // Expanded Drop / top-2: candidates per token

// ------------------------------------------------------------------ router
struct RouterArgs {
  const void* x;          // [T, d] fp32 or bf16 (ignored when logits_in is set)
  const float* W_g;       // [N, d]
  const float* b_g;       // [N] or null
  const float* logits_in; // [T, N] or null: route these logits instead of x W_g^T
  float* logits_out;      // [T, N] or null: only compute and store the logits
  int T, d, N;
  int x_is_bf16;
  // routing outputs
  int32_t* expert_id;     // [T]
  float* gate;            // [T]
  float* P_part;          // [R, N]  per-CTA sums of the probabilities
  int32_t* hist;          // [R, N]  per-CTA expert histograms (scanned in place later)
  int32_t* local_rank;    // [T]     rank of the token among same-expert tokens of its CTA
  int32_t* ctrl;          // control words (zeroed by CTA 0)
  // Expanded Drop: n_cand > 1 also stores each token's first n_cand experts
  // by logit (lowest index first on ties) and their probabilities
  int n_cand;
  int32_t* cand;          // [T][kMaxCand]
  float* cand_p;          // [T][kMaxCand]
  // top-2 (n_cand == 2): histogram and in-group ranks of every token's
  // second choice cand[1], like hist / local_rank for the first; or null
  int32_t* hist2;         // [R, N]
  int32_t* local_rank2;   // [T]
  // expert choice: every probability, transposed (expert e's scores of all
  // tokens contiguous), or null
  float* probs_t;         // [N, T]
  // Router split along K (few tokens, long d_model): the tensor-core router
  // writes each K range's logit sums to part_out [split][T][N] (no bias, no
  // routing); the FFMA router's kernel then routes sum_p parts_in[p] + b_g,
  // parts in order.
  float* part_out;
  const float* parts_in;
  int n_parts;
};

// A token's first kMaxCand experts by logit, descending, lowest index first
// among equal logits, in one pass over its N logits (at(i) is logit i):
// insertion into a sorted list of kMaxCand.  A logit goes in above the first
// entry it strictly exceeds (an equal logit stays behind the earlier index)
// and every entry from there on moves down one place.  cand[0] is the top-1
// expert (the first maximum).
template <typename At>
__device__ __forceinline__ void topk_candidates(At at, int N, int (&cand)[kMaxCand],
                                                float (&cv)[kMaxCand]) {
#pragma unroll
  for (int q = 0; q < kMaxCand; ++q) {
    cand[q] = -1;
    cv[q] = 0.f;
  }
  for (int i = 0; i < N; ++i) {
    float nv = at(i);
    int ni = i;
    bool moved = false;
#pragma unroll
    for (int q = 0; q < kMaxCand; ++q) {
      if (moved || cand[q] < 0 || nv > cv[q]) {
        const float tv = cv[q];
        const int ti = cand[q];
        cv[q] = nv;
        cand[q] = ni;
        nv = tv;
        ni = ti;
        moved = true;
      }
    }
  }
}
// Adds one epilogue warp's 32-row x 32-token block of an expert output into
// y with 16-byte atomic adds (several slots may add into one token's row).
// On entry lane l holds rows r0 + l for tokens c0 .. c0 + 31 in v (column
// jj in v[jj / 16][jj % 16]); token and gate of column c0 + l are in tk32 /
// gv32.  The block is transposed by shuffles so that each lane adds 4
// consecutive rows of one token: 8 vector adds per lane instead of 32
// scalar ones.  ld: y's row stride; rows: rows of y (a multiple of 4).
__device__ __forceinline__ void add_block_v4(float (&v)[2][16], int tk32, float gv32, float* y,
                                             int ld, int r0, int rows, int c0, int nv,
                                             int lane) {
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) v[jj >> 4][jj & 15] *= __shfl_sync(0xffffffffu, gv32, jj);
  const int rg = lane & 7;        // this lane's 4-row group
  const int part = lane >> 3;     // which of 4 tokens per round it takes
#pragma unroll
  for (int k = 0; k < 8; ++k) {   // round k: tokens 4k .. 4k + 3
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float got = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float t = __shfl_sync(0xffffffffu, v[(4 * k + m) >> 4][(4 * k + m) & 15], rg * 4 + i);
        if (part == m) got = t;
      }
      w[i] = got;
    }
    const int jj = 4 * k + part;
    const int tj = __shfl_sync(0xffffffffu, tk32, jj);
    const int r = r0 + 4 * rg;
    if (c0 + jj < nv && r < rows)
      atomicAdd(reinterpret_cast<float4*>(y + (size_t)tj * (size_t)ld + r),
                make_float4(w[0], w[1], w[2], w[3]));
  }
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
// bf16 layers with N <= kMaxExpertsTc: W_g split into three bf16 pieces
// [3][n_mma][d] (rows >= N zero), then the tensor-core router over them.
int router_tc_n_mma(int N);
cudaError_t launch_split_wg(const float* W_g, __nv_bfloat16* pieces, int N, int d,
                            cudaStream_t s);
// ksplit > 1 (N <= 128 only): K ranges over blockIdx.y, sums to a.part_out.
cudaError_t launch_router_tc(const RouterArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             int* status, cudaStream_t s, bool pdl = false, int ksplit = 1);

// ------------------------------------------------------- scan / tile lists
struct ScanArgs {
  int32_t* hist;          // [R, N] in: histograms; out: exclusive per-expert bases
  const float* P_part;    // [R, N]
  int R, N, T, C;
  int32_t* counts;        // [N] out: expert_counts
  float* P_sum;           // [N] out: sum over tokens of the probability of expert i
  int32_t* expert_start;  // [N + 1] out: exclusive prefix of counts
  float* aux_loss;        // [1] out
  int2* entries;          // [N * ceil(C / BN)] out: (expert, token tile) work items
  int BN;                 // token tile of the expert GEMMs
  int32_t* ctrl;          // ctrl[0] done counter, ctrl[1] number of entries
  int32_t* split_cnt;     // [n_split_cnt] zeroed for the expert GEMMs' tail split, or null
  int n_split_cnt;
  // 1: the scan stores counts / probability sums only; finish_experts (prefix,
  // work list, L_aux) runs in an extra CTA of the slot-assignment kernel
  int defer_finish;
  // filled slots per expert for the work list (Expanded Drop), or null:
  // min(counts, C)
  const int32_t* kept;
  // top-2: the second choices' histograms; CTAs N .. 2N-1 scan them into
  // per-expert bases after the first choices and their totals into counts2;
  // finish_experts then fills kept_out = min(C, min(counts, C) + counts2)
  int32_t* hist2;
  int32_t* counts2;
  int32_t* kept_out;
  // expert choice: every expert keeps kept_all tokens (> 0), or 0
  int kept_all;
  // zeroed by the scan's CTAs (expert choice: the per-token expert counts
  // the selection then increments), or null
  int32_t* zero_buf;
  int n_zero;
};
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s, bool pdl = false);

// --------------------------------------------- slots, lists, dispatch
struct AssignArgs {
  int T, N, C, d;
  int elem_bytes;              // 2 (bf16) or 4 (fp32)
  int mode;                    // SWITCH_MOE_TOKEN_ORDER / SWITCH_MOE_GATE_PRIORITY
  const int32_t* expert_id;
  const float* gate;
  const int32_t* bases;        // [R, N] scanned histograms
  const int32_t* local_rank;   // [T]
  const int32_t* counts;       // [N]
  const int32_t* expert_start; // [N + 1]
  int32_t* sorted_list;        // [T] tokens grouped by expert, token order within
  int32_t* slot;               // [T]
  uint8_t* drop;               // [T]
  const void* x;               // [T, d]
  void* xbuf;                  // [N * C, d]
  int32_t* tok_of_slot;        // [N * C] token of each filled slot, or null
  float* y;                    // [T, d] fp32: rows of dropped tokens zeroed, or null
  int* status;
  // top-2 (topk == 2, token order): each token's two choices come from
  // cand / cand_p (choice 0 = top-1); expert_id and gate above are unused;
  // outputs [T, 2] go to eid_out / gate_out and slot / drop; tok_of_slot
  // holds 2 t + choice; y rows are all zeroed (both choices add into y)
  int topk;
  int renorm;                  // gates renormalised over the two choices
  const int32_t* cand;         // [T][kMaxCand]
  const float* cand_p;         // [T][kMaxCand]
  const int32_t* bases2;       // [R, N] scanned second-choice histograms
  const int32_t* local_rank2;  // [T]
  int32_t* eid_out;            // [T, 2]
  float* gate_out;             // [T, 2]
  float* slot_gate;            // [N * C] gate of each filled slot, for the combine
};
// Token order: slot, drop and the dispatch copy in one pass.
// Gate priority: only the per-expert token lists.
// finish (token order, or null): the scan's arguments when it ran with
// defer_finish; one extra CTA then completes the pass over experts.
cudaError_t launch_assign(const AssignArgs& a, const ScanArgs* finish, cudaStream_t s,
                          bool pdl = false);
// Gate priority: per-expert ranking by (gate desc, token asc); slot and drop.
cudaError_t launch_gate_select(const AssignArgs& a, cudaStream_t s, bool pdl = false);
// Copy kept rows x[t] -> xbuf[e * C + slot[t]] (gate-priority path).
cudaError_t launch_dispatch(const AssignArgs& a, cudaStream_t s, bool pdl = false);

// ------------------------------------------- Expanded Drop, passes 2..k
struct ExpandArgs {
  int T, N, C, d, elem_bytes;
  int k;                       // candidates per token (2..kMaxCand)
  const int32_t* cand;         // [T][kMaxCand]
  const float* cand_p;         // [T][kMaxCand]
  const int32_t* counts;       // [N] top-1 counts: pass 1 filled min(counts, C) slots
  int32_t* open;               // [T] scratch: tokens still unplaced, in token order
  int32_t* moved;              // [T] out: tokens placed by passes 2..k
  int32_t* n_moved;            // [1] out: their number
  int32_t* used;               // [N] out: filled slots after the last pass
  int32_t* expert_id;          // [T] rewritten for moved tokens
  float* gate;
  int32_t* slot;
  uint8_t* drop;
  int32_t* tok_of_slot;        // [N * C] or null
  const void* x;               // null: routing only
  void* xbuf;
};
// ------------------------------------------------------- expert choice
struct ExpertChoiceArgs {
  int T, N, C, d, elem_bytes;
  const float* probs_t;        // [N, T] router probabilities, transposed
  int32_t* chosen_token;       // [N, C] out: each expert's tokens, best first; -1 past T
  float* chosen_gate;          // [N, C] out: their scores (0 past T)
  int32_t* per_token;          // [T] out: experts that took each token (zeroed by the scan)
  int32_t* tok_of_slot;        // [N * C] or null
  float* slot_gate;            // [N * C] or null
  const void* x;               // null: routing only
  void* xbuf;
  float* y;                    // [T, d]: zeroed for the combine's adds, or null
  int* status;
};
// One CTA per expert: the expert's min(C, T) best tokens by (score desc,
// token asc) -- radix select of the C-th key, then a sort of the kept keys --
// their slots, gates and dispatch copies; one extra CTA runs finish_experts
// (fin.kept_all = min(C, T)).
cudaError_t launch_expert_select(const ExpertChoiceArgs& a, const ScanArgs& fin, cudaStream_t s,
                                 bool pdl);

// Passes 2..k in one CTA, after the top-1 pass placed its tokens: the
// unplaced tokens in token order try their next candidate while it has
// room; then finish_experts over the final filled slots (fin.kept = used).
cudaError_t launch_expand(const ExpandArgs& a, const ScanArgs& fin, cudaStream_t s, bool pdl);
// Dispatch copies of the moved tokens' rows.
cudaError_t launch_expand_dispatch(const ExpandArgs& a, cudaStream_t s, bool pdl);

// ------------------------------------------------------- expert GEMMs
// D[e, m, c] = sum_k A[e * M + m, k] * B[e * rows + nt * BN + c, k] for the
// (expert, token tile) work items; m spans M in 128-row tiles.
struct GemmArgs {
  int M, K;                 // rows of A per expert, reduction length
  int rows_per_expert;      // rows of B (and of the output) per expert
  int BN;                   // token tile (tensor path: box rows, multiple of 16, <= 256)
  int m_tiles, k_blocks, ksplit;
  int num_b;                // 1: B0 only; 2: B0 + B1 (hi + lo halves of a split operand)
  int stages;
  const int2* entries;      // work items, or null for one dense problem (e = 0)
  const int32_t* n_entries; // device count of work items (entries != null)
  int n_entries_dense;      // count when entries == null
  const int32_t* counts;    // kept_e = min(counts[e], cap); null: every row kept
  int cap;
  int epi;                  // 0: relu -> (bf16 hi, bf16 lo) or fp32; 1: fp32 store;
                            // 2: combine (tensor path): y[tok] = g_tok * D (+ y[tok])
  void* out0;               // epi 2: y [T, M] fp32
  void* out1;
  int ldo;                  // output row stride (elements)
  size_t split_stride;      // elements between the outputs of successive K splits
  // epi 2: token of every filled slot, gates, scale flag, accumulate into y
  const int32_t* tok_of_slot;   // [N * C]
  const float* gate;            // [T]
  int gate_multiply;
  // 0: store; 1: add to y (one writer per row); 2: several slots add into
  // one row (top-2, expert choice): atomic adds, each slot's gate from
  // slot_gate
  int y_acc;
  const float* slot_gate;   // [N * C], y_acc 2
  // Tensor path, ksplit == 1: when the last wave of tiles is less than half
  // full, its tiles are cut along K into pieces that run on the idle CTAs;
  // the pieces leave fp32 partials and the last piece of each 32-row slice
  // to finish sums them in piece order.  null part: no tail split.
  float* part;              // [part_units][kTileM * BN]
  int part_units;
  int32_t* split_cnt;       // [4 * part_units]: zero on entry, left zero on exit
  int* status;
  int grid;
  size_t smem_bytes;
};
// tcgen05 tensor-core path (bf16 operands), TMA-fed.
cudaError_t launch_gemm_tc(const GemmArgs& g, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                           const CUtensorMap& tmB1, cudaStream_t s, bool pdl = false);
// exact-fp32 path (SIMT FFMA) for dtype fp32; A, B are fp32 device pointers.
cudaError_t launch_gemm_simt(const GemmArgs& g, const float* A, const float* B, cudaStream_t s,
                             bool pdl = false);
int gemm_tc_max_stages(int BN, int num_b);
size_t gemm_tc_smem_bytes(int BN, int num_b, int stages);

// ------------------------------------------------------- fused expert FFN
// GEMM 1 (+ ReLU, H hi + lo) and GEMM 2 (+ combine into y) of the routed
// experts in one persistent launch (tensor path, token tile <= 128).
constexpr int kFfnMaxBlocks = 256;   // blocks of work items in the schedule
struct FfnArgs {
  int C, BN;                  // slots per expert, token tile
  int d, F;                   // d_model, d_ff
  int m1, kb1;                // GEMM 1: 128-row tiles over F, 64-wide K blocks over d
  int m2, kb2;                // GEMM 2: 128-row tiles over d, 64-wide K blocks over F
  const int2* entries;        // work items (expert, token tile)
  const int32_t* n_entries;   // device count of work items
  const int32_t* counts;      // kept_e = min(counts[e], cap)
  int cap;
  int eb;                     // work items per schedule block
  int32_t* dep;               // [work items] GEMM 1 slices stored; zero on entry
  int32_t* sched;             // [1] next unit to claim; zero on entry
  const void* W1;             // [N, F, d] (L2 prefetch hint before the dependency wait)
  int n_experts;
  __nv_bfloat16* H0;          // [N * C, F] hi
  __nv_bfloat16* H1;          // [N * C, F] lo
  float* y;                   // [T, d]
  const int32_t* tok_of_slot; // [N * C] token of each filled slot
  const float* gate;          // [T] (y_acc 0, 1)
  int gate_multiply;
  // 0: store; 1: add to y (one writer per row); 2: several slots add into
  // one row (top-2, expert choice): atomic adds, each slot's gate from
  // slot_gate
  int y_acc;
  const float* slot_gate;     // [N * C], y_acc 2
  float* part;                // tail split partials [part_units][128 * BN], or null
  int part_units;
  int32_t* split_cnt;         // [4 * part_units]
  int stages;
  int* status;
  int grid;
  size_t smem_bytes;
};
int ffn_tc_stages(int BN);
size_t ffn_tc_smem_bytes(int BN, int stages);
cudaError_t launch_ffn_tc(const FfnArgs& a, const CUtensorMap& tmW1, const CUtensorMap& tmX,
                          const CUtensorMap& tmW2, const CUtensorMap& tmH0,
                          const CUtensorMap& tmH1, cudaStream_t s, bool pdl);

// ------------------------------------------------------- combine
struct CombineArgs {
  int T, d, C, ksplit;
  int gate_multiply;
  int topk;                 // choices per token (expert_id, gate, slot are [T, topk])
  const int32_t* expert_id;
  const float* gate;
  const int32_t* slot;
  const float* O;           // [ksplit][N * C, d] fp32 partial expert outputs
  size_t split_stride;      // elements between K-split partials
  const float* S;           // [T, d] shared-expert output or null
  float* y;                 // [T, d]
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl = false);

// Combine by slots (expert choice on the paths without the fused combine):
// y[tok(slot)] += g(slot) * sum_k O_k[slot] for every filled slot, and
// y[t] += S[t] -- atomic adds into a y the selection zeroed.
struct SlotCombineArgs {
  int T, N, C, d, ksplit, kept;   // kept: filled slots per expert
  int gate_multiply;
  const int32_t* tok_of_slot;     // [N * C]
  const float* slot_gate;         // [N * C]
  const float* O;                 // [ksplit][N * C, d]
  size_t split_stride;
  const float* S;                 // [T, d] or null
  float* y;
};
cudaError_t launch_combine_slots(const SlotCombineArgs& a, cudaStream_t s, bool pdl = false);

// ------------------------------------------------------- backward
// Strided batched fp32 GEMM: C_b[m, n] (+)= sum_k A_b[m, k] B_b[n, k], with
// A_b[m, k] = A[b a_b + m a_m + k a_k] (B and C likewise); per-batch counts
// (null: the full M, N, K) limit batch b's rows and reduction.
struct BGemmArgs {
  int M, N, K, batches;
  const int32_t* mcount;
  const int32_t* ncount;
  const int32_t* kcount;
  size_t a_b, a_m, a_k;
  size_t b_b, b_n, b_k;
  size_t c_b, c_m, c_n;
  float* C;
  int accumulate;
  // > 0: batch b takes the reduction range [b k_chunk, (b + 1) k_chunk) of K
  // (its partial result goes to C + b c_b; launch_bwd_sum adds the parts)
  int k_chunk;
};
cudaError_t launch_bgemm(const BGemmArgs& g, const void* A, bool a_bf16, const void* B,
                         bool b_bf16, cudaStream_t s);

struct BwdArgs {
  int T, N, C, d;
  int gate_multiply;
  float aux_coef;
  const int32_t* expert_id;   // [T] forward's top-1 expert
  const int32_t* slot;        // [T] forward's slot, -1 dropped
  const int32_t* counts;      // [N] forward's expert_counts (f_i)
  const float* gate;          // [T]
  const float* dy;            // [T, d] upstream gradient of y
  float* Xg;                  // [N C, d] dispatched rows (fp32)
  float* dO;                  // [N C, d] gradient of each slot's expert output
  float* O;                   // [N C, d] each slot's expert output E(x)
  float* dX;                  // [N C, d] gradient of each slot's input row
  float* dx;                  // [T, d] out
  float* dgate;               // [T] gradient of the gate
  float* L;                   // [T, N] logits without the bias in, router logit gradient out
  const float* b_g;           // [N] or null
  int32_t* tok;               // [N C] token of each slot
};
cudaError_t launch_bwd_gather(const BwdArgs& a, const void* x, bool x_bf16, cudaStream_t s);
cudaError_t launch_bwd_relu(float* H, const int32_t* counts, int C, int F, int N,
                            cudaStream_t s);
cudaError_t launch_bwd_mask(float* dH, const float* H, const int32_t* counts, int C, int F,
                            int batches, cudaStream_t s);
cudaError_t launch_bwd_scatter(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_router(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_colsum(const float* dl, float* out, int T, int N, cudaStream_t s);
// out[i] = sum_p parts[p n + i], parts in order (K-split partial results).
cudaError_t launch_bwd_sum(const float* parts, int n_parts, size_t n, float* out, cudaStream_t s);

// status word of the current device (see switch_moe_sync_status)
int* device_status_ptr();

cudaError_t launch_selftest_wait(int* status, unsigned long long timeout_ns, cudaStream_t s);

}  // namespace smoe
