// Capacity-limited slot assignment, overflow, dispatch into the per-expert
// buffer, and the auxiliary-loss reduction.
//
// Sources: "Top-1 路由 (Top-1 Routing)" (compassingai.com), Token Dropping
// section (an expert takes at most capacity tokens; the rest skip it) and
// load-balancing section (L_aux = N * sum_i f_i P_i); Switch Transformer
// walk-through (personwebsite.pages.dev/moe-switch), expert-capacity section;
// "MoE 专家容量因子与 Token 丢弃" (wiblog.cn): capacity turns routing into a
// fixed [N, C, d] buffer (section on where capacity comes from), and the
// overflow section plus the token-path flowchart (nodes D -> F): once every
// score is known, an over-full expert keeps its highest-weight tokens.
//
// Dispatch: each kept row is copied x[t] -> buffer[e, slot] by two TMA bulk
//   copies through shared memory (the load starts before the slot is known).
// Token order:   slot(t) = #{t' < t : e(t') = e(t)}; kept iff slot < C.
//   The router already produced, per CTA of 32 tokens, an expert histogram
//   and each token's rank inside its CTA; scan_kernel turns the histograms
//   into per-expert exclusive prefixes over CTAs (one CTA per expert), so
//   slot = prefix[cta(t)][e] + rank(t) -- integer work, bit-exact.
// Gate priority: tokens of one expert ordered by (gate desc, token asc);
//   slot = rank in that order; kept iff rank < C.  One CTA per expert sorts
//   the 64-bit keys (~gate_bits << 32 | token) in shared memory; experts
//   with more tokens than fit first radix-select the C-th smallest key.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kScanThreads = 256;

// Exclusive scan of one int per thread across the block (up to 1024 threads).
__device__ int block_exclusive_scan(int v, int* total, int* sh /*[32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? sh[lane] : 0;
    int winc = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, winc, off);
      if (lane >= off) winc += o;
    }
    sh[lane] = winc - w;             // exclusive prefix of warp sums
    if (lane == 31) sh[32] = winc;   // block total
  }
  __syncthreads();
  int res = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return res;
}

// Fixed-shape tree sum (reproducible run to run).
template <typename F>
__device__ F block_sum(F v, F* sh /*[32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  F r = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += sh[w];
  __syncthreads();
  return r;   // valid in thread 0
}

// After every expert's count and probability sum are stored: exclusive
// prefix of the counts, the GEMM work items (expert, token tile) in expert
// order, L_aux, and zeroed counters for the expert GEMMs.  Run by one CTA
// of kScanThreads threads: the last scan CTA to finish, or (token order)
// an extra CTA of the slot-assignment kernel, off the scan's critical path.
__device__ void finish_experts(const ScanArgs& a, int* sh_i, double* sh_d) {
  const int tid = threadIdx.x;
  // Each thread owns a contiguous run of up to 4 experts.
  const int per_e = (a.N + (int)blockDim.x - 1) / (int)blockDim.x;   // <= 4 for N <= 1024
  const int e0 = min(a.N, tid * per_e), e1 = min(a.N, e0 + per_e);
  int c_loc = 0, t_loc = 0;
  double aux_loc = 0.0;
  int cv[4], nv[4];   // this thread's counts and token tiles, loaded once
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = e0 + j;
    cv[j] = 0;
    nv[j] = 0;
    if (i < e1) {
      const int c = __ldcg(a.counts + i);
      const float p = __ldcg(a.P_sum + i);
      int kept = a.kept ? __ldcg(a.kept + i) : min(c, a.C);
      if (a.counts2) kept = min(a.C, kept + __ldcg(a.counts2 + i));   // top-2: then choice 1
      if (a.kept_all > 0) kept = a.kept_all;                          // expert choice
      if (a.kept_out) a.kept_out[i] = kept;
      cv[j] = c;
      nv[j] = (kept + a.BN - 1) / a.BN;
      c_loc += c;
      t_loc += nv[j];
      aux_loc += (double)c * (double)p;
    }
  }
  int c_tot, t_tot;
  int c_run = block_exclusive_scan(c_loc, &c_tot, sh_i);
  int t_run = block_exclusive_scan(t_loc, &t_tot, sh_i);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = e0 + j;
    if (i < e1) {
      a.expert_start[i] = c_run;
      c_run += cv[j];
      for (int q = 0; q < nv[j]; ++q) a.entries[t_run + q] = make_int2(i, q);
      t_run += nv[j];
    }
  }
  const double aux = block_sum<double>(aux_loc, sh_d);
  if (a.split_cnt)
    for (int i = tid; i < a.n_split_cnt; i += blockDim.x) a.split_cnt[i] = 0;
  if (tid == 0) {
    a.expert_start[a.N] = c_tot;
    a.ctrl[1] = t_tot;
    const double T = (double)a.T;
    a.aux_loss[0] = (float)((double)a.N * aux / (T * T));  // N * sum (c_i / T)(P_i / T)
    a.ctrl[0] = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  __shared__ int sh_i[33];
  __shared__ float sh_f[32];
  __shared__ double sh_d[32];
  __shared__ int is_last;
  grid_dep_wait();
  grid_dep_launch();
  if (a.zero_buf)
    for (int i = blockIdx.x * kScanThreads + threadIdx.x; i < a.n_zero;
         i += gridDim.x * kScanThreads)
      a.zero_buf[i] = 0;
  // CTAs N .. 2N-1 (top-2): the second choices' histograms, no probabilities
  const bool second = blockIdx.x >= a.N;
  const int e = second ? blockIdx.x - a.N : blockIdx.x, tid = threadIdx.x;
  int32_t* hist = second ? a.hist2 : a.hist;
  const int per = (a.R + kScanThreads - 1) / kScanThreads;
  const int r0 = min(a.R, tid * per), r1 = min(a.R, r0 + per);
  int cnt = 0;
  float ps = 0.f;
  for (int r = r0; r < r1; ++r) {
    cnt += hist[(size_t)r * a.N + e];
    if (!second) ps += a.P_part[(size_t)r * a.N + e];
  }
  int total;
  int run = block_exclusive_scan(cnt, &total, sh_i);
  for (int r = r0; r < r1; ++r) {
    const size_t i = (size_t)r * a.N + e;
    const int v = hist[i];
    hist[i] = run;
    run += v;
  }
  const float psum = block_sum<float>(ps, sh_f);
  if (tid == 0) {
    if (second) {
      a.counts2[e] = total;
    } else {
      a.counts[e] = total;
      a.P_sum[e] = psum;
    }
  }
  if (a.defer_finish) return;   // the slot-assignment kernel runs finish_experts
  if (tid == 0) {
    __threadfence();
    is_last = (atomicAdd(&a.ctrl[0], 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  finish_experts(a, sh_i, sh_d);
}

// Copy one row of `bytes` (a multiple of 16) with the lanes of a warp.
__device__ __forceinline__ void copy_row(const void* __restrict__ src, void* __restrict__ dst,
                                         int bytes, int lane) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  const int nv = bytes >> 4;
  int v = lane;
  for (; v + 64 < nv; v += 96) {    // three independent 16-byte loads in flight per lane
    uint4 a0 = __ldg(s + v), a1 = __ldg(s + v + 32), a2 = __ldg(s + v + 64);
    d[v] = a0; d[v + 32] = a1; d[v + 64] = a2;
  }
  for (; v < nv; v += 32) d[v] = __ldg(s + v);
}

// Zero one fp32 row of d (a multiple of 8) values: the MoE-branch output of
// a dropped token, which skips every expert.
__device__ __forceinline__ void zero_row(float* row, int d, int lane) {
  float4* r = reinterpret_cast<float4*>(row);
  for (int v = lane; v < (d >> 2); v += 32) r[v] = make_float4(0.f, 0.f, 0.f, 0.f);
}

constexpr int kRowWarps = 8;   // tokens per CTA in the per-token kernels

// Rows up to this size are staged through shared memory by TMA bulk copies;
// longer rows use the vector copy.
constexpr uint32_t kStageRowMax = 16384;

// Bounded wait on a bulk copy's mbarrier (one thread); false on timeout.
__device__ __forceinline__ bool row_wait(uint64_t* bar, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 0; it < kWaitMaxIters; ++it) {
    if (mbar_try_wait(bar, 0u)) return true;
    if ((it & 31u) == 31u && globaltimer_ns() - t0 > kWaitTimeoutNs) break;
  }
  atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
  return false;
}

// Dispatch of token t's row into the expert buffer (row `dst_row`, or no copy
// when dst_row < 0), staged through this warp's slot of shared memory:
// the TMA load was started by stage_row_begin before the destination was
// known; lane 0 waits for it and issues the TMA store.
__device__ __forceinline__ void stage_row_begin(const AssignArgs& a, uint8_t* buf, uint64_t* bar,
                                                int t, uint32_t rb, int lane) {
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, rb);
    bulk_load(buf, static_cast<const char*>(a.x) + (size_t)t * rb, rb, bar);
  }
}
// A second destination (e2, dst_row2 >= 0) takes the same row: top-2.
__device__ __forceinline__ void stage_row_end(const AssignArgs& a, uint8_t* buf, uint64_t* bar,
                                              int e, int dst_row, uint32_t rb, int lane,
                                              int e2 = 0, int dst_row2 = -1) {
  if (lane == 0) {
    // the load must land before the CTA may exit, copied or not
    if (row_wait(bar, a.status) && (dst_row >= 0 || dst_row2 >= 0)) {
      fence_proxy_async_smem();
      char* xb = static_cast<char*>(a.xbuf);
      if (dst_row >= 0) bulk_store(xb + ((size_t)e * a.C + dst_row) * rb, buf, rb);
      if (dst_row2 >= 0) bulk_store(xb + ((size_t)e2 * a.C + dst_row2) * rb, buf, rb);
      bulk_commit();
      bulk_wait_read();
    }
  }
}

// Top-2, token order: choice 0 takes slot bases[g][e0] + rank, as in top-1;
// choice 1 queues behind every first choice its expert kept:
// slot min(counts[e1], C) + bases2[g][e1] + rank2.  Each is kept iff its
// slot < C.  The gates are the two probabilities, or renormalised over the
// pair.  The x row goes to both kept slots; y is zeroed for the atomic
// accumulation of the two outputs.
__device__ __forceinline__ void assign_top2(const AssignArgs& a, int t, uint8_t* buf,
                                            uint64_t* bar, uint32_t rb, bool staged, int lane) {
  const size_t g = (size_t)(t / kRouterTM) * a.N;
  const int e0 = a.cand[(size_t)t * kMaxCand], e1 = a.cand[(size_t)t * kMaxCand + 1];
  const int s0 = a.bases[g + e0] + a.local_rank[t];
  const int s1 = min(a.counts[e1], a.C) + a.bases2[g + e1] + a.local_rank2[t];
  const bool k0 = s0 < a.C, k1 = s1 < a.C;
  if (lane == 0) {
    float g0 = a.cand_p[(size_t)t * kMaxCand], g1 = a.cand_p[(size_t)t * kMaxCand + 1];
    if (a.renorm) {
      const float z = g0 + g1;
      g0 = g0 / z;
      g1 = g1 / z;
    }
    a.eid_out[2 * (size_t)t] = e0;
    a.eid_out[2 * (size_t)t + 1] = e1;
    a.gate_out[2 * (size_t)t] = g0;
    a.gate_out[2 * (size_t)t + 1] = g1;
    a.slot[2 * (size_t)t] = k0 ? s0 : -1;
    a.slot[2 * (size_t)t + 1] = k1 ? s1 : -1;
    a.drop[2 * (size_t)t] = k0 ? 0 : 1;
    a.drop[2 * (size_t)t + 1] = k1 ? 0 : 1;
    if (a.xbuf && a.tok_of_slot) {
      if (k0) {
        a.tok_of_slot[(size_t)e0 * a.C + s0] = t;
        a.slot_gate[(size_t)e0 * a.C + s0] = g0;
      }
      if (k1) {
        a.tok_of_slot[(size_t)e1 * a.C + s1] = t;
        a.slot_gate[(size_t)e1 * a.C + s1] = g1;
      }
    }
  }
  if (staged) {
    stage_row_end(a, buf, bar, e0, k0 ? s0 : -1, rb, lane, e1, k1 ? s1 : -1);
  } else if (a.xbuf) {
    const char* src = static_cast<const char*>(a.x) + (size_t)t * rb;
    char* xb = static_cast<char*>(a.xbuf);
    if (k0) copy_row(src, xb + ((size_t)e0 * a.C + s0) * rb, (int)rb, lane);
    if (k1) copy_row(src, xb + ((size_t)e1 * a.C + s1) * rb, (int)rb, lane);
  }
  if (a.y) zero_row(a.y + (size_t)t * a.d, a.d, lane);
}

__global__ void __launch_bounds__(kRowWarps * 32) assign_kernel(AssignArgs a, ScanArgs sa) {
  extern __shared__ __align__(128) uint8_t rowbuf[];   // [kRowWarps][rb] when staged
  __shared__ __align__(8) uint64_t rowbar[kRowWarps];
  grid_dep_wait();
  grid_dep_launch();
  if (sa.defer_finish && blockIdx.x == gridDim.x - 1) {   // the extra CTA
    __shared__ int sh_i[33];
    __shared__ double sh_d[32];
    finish_experts(sa, sh_i, sh_d);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + warp;
  if (t >= a.T) return;
  const uint32_t rb = (uint32_t)a.d * (uint32_t)a.elem_bytes;
  const bool staged = a.mode == SWITCH_MOE_TOKEN_ORDER && a.xbuf && rb <= kStageRowMax;
  uint8_t* buf = rowbuf + (size_t)warp * rb;
  if (staged) stage_row_begin(a, buf, &rowbar[warp], t, rb, lane);   // x row is known already
  if (a.topk == 2) {
    assign_top2(a, t, buf, &rowbar[warp], rb, staged, lane);
    return;
  }
  const int e = a.expert_id[t];
  const int s = a.bases[(size_t)(t / kRouterTM) * a.N + e] + a.local_rank[t];
  if (a.mode == SWITCH_MOE_TOKEN_ORDER) {
    const bool kept = s < a.C;
    if (lane == 0) {
      a.slot[t] = kept ? s : -1;
      a.drop[t] = kept ? 0 : 1;
      if (kept && a.xbuf && a.tok_of_slot) a.tok_of_slot[(size_t)e * a.C + s] = t;
    }
    if (staged) {
      stage_row_end(a, buf, &rowbar[warp], e, kept ? s : -1, rb, lane);
    } else if (kept && a.xbuf) {   // no buffer when only routing (route_from_logits)
      copy_row(static_cast<const char*>(a.x) + (size_t)t * rb,
               static_cast<char*>(a.xbuf) + ((size_t)e * a.C + s) * rb, (int)rb, lane);
    }
    if (!kept && a.y) zero_row(a.y + (size_t)t * a.d, a.d, lane);
  } else if (lane == 0) {
    a.sorted_list[a.expert_start[e] + s] = t;
  }
}

__global__ void __launch_bounds__(kRowWarps * 32) dispatch_kernel(AssignArgs a) {
  extern __shared__ __align__(128) uint8_t rowbuf[];
  __shared__ __align__(8) uint64_t rowbar[kRowWarps];
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRowWarps + warp;
  if (t >= a.T) return;
  const uint32_t rb = (uint32_t)a.d * (uint32_t)a.elem_bytes;
  const bool staged = rb <= kStageRowMax;
  uint8_t* buf = rowbuf + (size_t)warp * rb;
  if (staged) stage_row_begin(a, buf, &rowbar[warp], t, rb, lane);
  const int s = a.slot[t];
  const int e = a.expert_id[t];
  if (s >= 0 && a.tok_of_slot && lane == 0) a.tok_of_slot[(size_t)e * a.C + s] = t;
  if (staged) {
    stage_row_end(a, buf, &rowbar[warp], e, s, rb, lane);
  } else if (s >= 0) {
    copy_row(static_cast<const char*>(a.x) + (size_t)t * rb,
             static_cast<char*>(a.xbuf) + ((size_t)e * a.C + s) * rb, (int)rb, lane);
  }
  if (s < 0 && a.y) zero_row(a.y + (size_t)t * a.d, a.d, lane);
}

// ------------------------------------------------- Expanded Drop passes
// After the top-1 pass, pass r (r = 2..k) runs over the tokens still
// unplaced, in token order: each tries its r-th candidate and takes that
// expert's next free slot while one is left ("MoE 专家容量因子与 Token 丢弃",
// wiblog.cn, inference section, on Capacity-Aware Inference's Expanded
// Drop: overflow tokens consider further experts of their candidate set).
// The processing expert's probability becomes the token's gate.
//
// One CTA of kExpandThreads: the unplaced tokens are few and every pass
// depends on the one before, so the CTA walks them in chunks of 1024.  In
// a chunk each token's slot is fill[e] + (same-candidate tokens of earlier
// warps) + (rank among its warp's same-candidate tokens); the last group of
// each expert in the chunk advances fill[e].  Tokens left over are compacted
// in order for the next pass.

constexpr int kExpandThreads = 1024;
constexpr int kExpandWarps = kExpandThreads / 32;

__global__ void __launch_bounds__(kExpandThreads, 1) expand_kernel(ExpandArgs a, ScanArgs fin) {
  extern __shared__ int xsm[];
  int* whist = xsm;                           // [kExpandWarps][N] group sizes
  int* fill = xsm + kExpandWarps * a.N;       // [N] filled slots
  __shared__ int sh_i[33];
  __shared__ double sh_d[32];
  grid_dep_wait();
  grid_dep_launch();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, N = a.N;
  for (int i = tid; i < kExpandWarps * N; i += kExpandThreads) whist[i] = 0;
  for (int e = tid; e < N; e += kExpandThreads) fill[e] = min(__ldcg(a.counts + e), a.C);
  // tokens the top-1 pass left unplaced, in token order: each warp owns a
  // contiguous run, read 32 tokens (one line) at a time, 8 lines in flight
  const int perw = ((a.T + kExpandWarps * 32 - 1) / (kExpandWarps * 32)) * 32;
  const int w0 = min(a.T, warp * perw), w1 = min(a.T, w0 + perw);
  const unsigned lt = (1u << lane) - 1u;
  int cw = 0;
  for (int b = w0; b < w1; b += 8 * 32) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = b + j * 32 + lane;
      v[j] = t < w1 ? __ldcg(a.slot + t) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) cw += __popc(__ballot_sync(0xffffffffu, v[j] < 0));
  }
  int n;
  int pos = __shfl_sync(0xffffffffu, block_exclusive_scan(lane == 0 ? cw : 0, &n, sh_i), 0);
  for (int b = w0; b < w1; b += 8 * 32) {
    int v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = b + j * 32 + lane;
      v[j] = t < w1 ? __ldcg(a.slot + t) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const unsigned m = __ballot_sync(0xffffffffu, v[j] < 0);
      if (v[j] < 0) a.open[pos + __popc(m & lt)] = b + j * 32 + lane;
      pos += __popc(m);
    }
  }
  int n_moved = 0;
  __syncthreads();
  for (int r = 1; r < a.k; ++r) {
    int n_next = 0;
    // the next chunk's tokens are loaded one chunk ahead: this chunk's
    // compaction writes only positions below them
    // (and their candidate and its probability once the token has arrived)
    int t_nx = tid < n ? __ldcg(a.open + tid) : -1;
    int e_nx = t_nx >= 0 ? __ldcg(a.cand + (size_t)t_nx * kMaxCand + r) : -1 - lane;
    float g_nx = t_nx >= 0 ? __ldcg(a.cand_p + (size_t)t_nx * kMaxCand + r) : 0.f;
    for (int c0 = 0; c0 < n; c0 += kExpandThreads) {
      const int t = t_nx, e = e_nx;
      const float gp = g_nx;
      const int i_nx = c0 + kExpandThreads + tid;
      t_nx = i_nx < n ? __ldcg(a.open + i_nx) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const bool leader = t >= 0 && (peers & lt) == 0;
      if (leader) whist[warp * N + e] = __popc(peers);
      __syncthreads();
      int s = 0, pre = 0;
      bool last = leader;
      if (t >= 0) {
        for (int w = 0; w < warp; ++w) pre += whist[w * N + e];
        s = fill[e] + pre + __popc(peers & lt);
        if (leader)
          for (int w = warp + 1; w < kExpandWarps && last; ++w) last = whist[w * N + e] == 0;
      }
      __syncthreads();   // every read of whist and fill is done
      e_nx = t_nx >= 0 ? __ldcg(a.cand + (size_t)t_nx * kMaxCand + r) : -1 - lane;
      g_nx = t_nx >= 0 ? __ldcg(a.cand_p + (size_t)t_nx * kMaxCand + r) : 0.f;
      if (leader) {
        if (last) fill[e] += pre + __popc(peers);
        whist[warp * N + e] = 0;
      }
      const bool placed = t >= 0 && s < a.C;
      if (placed) {
        a.slot[t] = s;
        a.drop[t] = 0;
        a.expert_id[t] = e;
        a.gate[t] = gp;
        if (a.tok_of_slot) a.tok_of_slot[(size_t)e * a.C + s] = t;
      }
      const bool stays = t >= 0 && !placed;
      // one scan for both lists: stays in the low half, placed in the high
      int tot;
      const int p = block_exclusive_scan((int)stays | ((int)placed << 16), &tot, sh_i);
      if (stays) a.open[n_next + (p & 0xffff)] = t;   // at or before position c0 + tid
      if (placed) a.moved[n_moved + (p >> 16)] = t;
      n_next += tot & 0xffff;
      n_moved += tot >> 16;
    }
    n = n_next;
    __syncthreads();
    for (int e = tid; e < N; e += kExpandThreads) fill[e] = min(fill[e], a.C);
    __syncthreads();
  }
  for (int e = tid; e < N; e += kExpandThreads) a.used[e] = fill[e];
  if (tid == 0) *a.n_moved = n_moved;
  __syncthreads();
  finish_experts(fin, sh_i, sh_d);   // fin.kept == a.used
}

// Rows of the tokens passes 2..k placed, one warp per row.
__global__ void __launch_bounds__(kRowWarps * 32) expand_dispatch_kernel(ExpandArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int n = __ldcg(a.n_moved);
  const uint32_t rb = (uint32_t)a.d * (uint32_t)a.elem_bytes;
  for (int j = blockIdx.x * kRowWarps + (threadIdx.x >> 5); j < n; j += gridDim.x * kRowWarps) {
    const int t = __ldcg(a.moved + j);
    const int e = __ldcg(a.expert_id + t), s = __ldcg(a.slot + t);
    copy_row(static_cast<const char*>(a.x) + (size_t)t * rb,
             static_cast<char*>(a.xbuf) + ((size_t)e * a.C + s) * rb, (int)rb, lane);
  }
}

constexpr int kSelThreads = 1024;

__device__ __forceinline__ unsigned long long gate_key(const AssignArgs& a, int t) {
  // gates are positive, so their bit patterns order like their values;
  // ascending key = descending gate, then ascending token
  const unsigned g = __float_as_uint(a.gate[t]);
  return ((unsigned long long)(~g) << 32) | (unsigned)t;
}

__device__ void bitonic_sort_asc(unsigned long long* k, int P) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int j = size >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = k[i], y = k[ixj];
          const bool up = (i & size) == 0;
          if ((x > y) == up) { k[i] = y; k[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// One radix-select step, run by warp 0: the first digit whose cumulative
// count over hist[0..255] reaches *krem (255 if none does); *krem drops by
// the count below it, and the digit joins *prefix / *mask at `shift`.  Each
// lane scans 8 bins; a warp scan and a ballot find the digit.
__device__ __forceinline__ void radix_pick(const int* hist, int shift, int* krem,
                                           unsigned long long* prefix,
                                           unsigned long long* mask, int* in_bin = nullptr) {
  const int lane = threadIdx.x & 31;
  int c[8], tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[lane * 8 + j];
    tot += c[j];
  }
  int inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  const int need = *krem;
  int below = inc - tot, dg = -1;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (dg < 0) {
      if (below + c[j] >= need) {
        dg = lane * 8 + j;
      } else {
        below += c[j];
      }
    }
  }
  const unsigned hit = __ballot_sync(0xffffffffu, dg >= 0);
  const int src = hit ? __ffs(hit) - 1 : 31;
  int digit = __shfl_sync(0xffffffffu, dg, src);
  int under = __shfl_sync(0xffffffffu, below, src);
  if (!hit) {   // no bin reaches krem: the last digit, everything below it counted
    digit = 255;
    under = __shfl_sync(0xffffffffu, inc, 31) - hist[255];
  }
  if (lane == 0) {
    *krem = need - under;
    *prefix |= (unsigned long long)digit << shift;
    *mask |= 255ull << shift;
    if (in_bin) *in_bin = hist[digit];
  }
}

__global__ void __launch_bounds__(kSelThreads) gate_select_kernel(AssignArgs a) {
  extern __shared__ unsigned long long sk[];   // [kGateSortMax]
  __shared__ int hist[256];
  __shared__ unsigned long long s_prefix, s_mask;
  __shared__ int s_krem, s_cnt;
  grid_dep_wait();
  grid_dep_launch();
  const int e = blockIdx.x, tid = threadIdx.x;
  const int n = a.counts[e];
  if (n == 0) return;
  const int32_t* list = a.sorted_list + a.expert_start[e];
  if (n <= kGateSortMax) {
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = tid; i < P; i += kSelThreads) sk[i] = (i < n) ? gate_key(a, list[i]) : ~0ull;
    __syncthreads();
    bitonic_sort_asc(sk, P);
    for (int i = tid; i < n; i += kSelThreads) {
      const int t = (int)(unsigned)(sk[i] & 0xffffffffull);
      const bool kept = i < a.C;
      a.slot[t] = kept ? i : -1;
      a.drop[t] = kept ? 0 : 1;
    }
    return;
  }
  // More tokens than fit: find the C-th smallest key by MSB-first radix
  // select (keys are unique), keep the keys at or below it, sort those.
  if (tid == 0) { s_prefix = 0ull; s_mask = 0ull; s_krem = a.C; }
  __syncthreads();
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const unsigned long long pre = s_prefix, msk = s_mask;
    for (int i = tid; i < n; i += kSelThreads) {
      const unsigned long long k = gate_key(a, list[i]);
      if ((k & msk) == pre) atomicAdd(&hist[(int)((k >> shift) & 255ull)], 1);
    }
    __syncthreads();
    if (tid < 32) radix_pick(hist, shift, &s_krem, &s_prefix, &s_mask);
    __syncthreads();
  }
  const unsigned long long thr = s_prefix;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  for (int i = tid; i < n; i += kSelThreads) {
    const unsigned long long k = gate_key(a, list[i]);
    if (k <= thr) {
      const int pos = atomicAdd(&s_cnt, 1);
      if (pos < kGateSortMax) sk[pos] = k;
    } else {
      const int t = list[i];
      a.slot[t] = -1;
      a.drop[t] = 1;
    }
  }
  __syncthreads();
  const int kept_n = min(s_cnt, kGateSortMax);   // == C
  int P = 1;
  while (P < kept_n) P <<= 1;
  for (int i = kept_n + tid; i < P; i += kSelThreads) sk[i] = ~0ull;
  __syncthreads();
  bitonic_sort_asc(sk, P);
  for (int i = tid; i < kept_n; i += kSelThreads) {
    const int t = (int)(unsigned)(sk[i] & 0xffffffffull);
    a.slot[t] = i;
    a.drop[t] = 0;
  }
}

// ------------------------------------------------------- expert choice
// Expert choice ("Top-1 路由 (Top-1 Routing)", compassingai.com,
// routing-paradigm table: each expert selects its top-K tokens; milestone
// table: Expert Choice Routing): expert e keeps the min(C, T) tokens with
// the highest router probability s[t, e], the lower token index first
// among equal scores, slot = rank.  Keys (~bits(s) << 32 | t) order that
// way (scores are >= 0, so their bit patterns order like their values).
__device__ __forceinline__ unsigned long long ec_key(const float* col, int t) {
  return ((unsigned long long)(~__float_as_uint(col[t])) << 32) | (unsigned)t;
}

__global__ void __launch_bounds__(kSelThreads) expert_select_kernel(ExpertChoiceArgs a,
                                                                    ScanArgs fin) {
  extern __shared__ unsigned long long sk[];   // [kGateSortMax]
  __shared__ int hist[256];
  __shared__ unsigned long long s_prefix, s_mask;
  __shared__ int s_krem, s_cnt;
  __shared__ int sh_i[33];
  __shared__ double sh_d[32];
  grid_dep_wait();
  grid_dep_launch();
  if (blockIdx.x == gridDim.x - 1) {   // the extra CTA: work list and L_aux
    finish_experts(fin, sh_i, sh_d);
    return;
  }
  const int e = blockIdx.x, tid = threadIdx.x, T = a.T;
  const int lane = tid & 31, warp = tid >> 5;
  const float* col = a.probs_t + (size_t)e * T;
  const int k = min(a.C, T);
  if (a.y) {   // rows t = e, e + N, ...: the combine adds every slot of a token into y
    const int nv = a.d >> 2;
    const int rows = (T - e + a.N - 1) / a.N;
    float4* y4 = reinterpret_cast<float4*>(a.y);
    for (size_t i = tid; i < (size_t)rows * nv; i += kSelThreads) {
      const size_t t = (size_t)e + (i / nv) * a.N;
      y4[t * nv + i % nv] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // keys in shared memory when they fit (T <= kGateSortMax), else re-read
  const bool cached = T <= kGateSortMax;
  if (cached)
    for (int i = tid; i < T; i += kSelThreads) sk[i] = ec_key(col, i);
  auto key_at = [&](int i) { return cached ? sk[i] : ec_key(col, i); };
  if (k < T) {
    // the k-th smallest key by MSB-first radix select (keys are unique);
    // histogram updates are aggregated per warp (scores share high bits).
    // The four score digits usually settle it: when the expert keeps every
    // key of the boundary score, the token digits are not needed.
    __shared__ int s_inbin;
    if (tid == 0) { s_prefix = 0ull; s_mask = 0ull; s_krem = k; s_cnt = 0; }
    __syncthreads();
    unsigned long long thr = 0ull;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      const unsigned long long pre = s_prefix, msk = s_mask;
      for (int i0 = 0; i0 < T; i0 += kSelThreads) {
        const int i = i0 + tid;
        int dg = -1;
        if (i < T) {
          const unsigned long long key = key_at(i);
          if ((key & msk) == pre) dg = (int)((key >> shift) & 255ull);
        }
        const unsigned peers = __match_any_sync(0xffffffffu, dg);
        if (dg >= 0 && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(&hist[dg], __popc(peers));
      }
      __syncthreads();
      if (tid < 32) radix_pick(hist, shift, &s_krem, &s_prefix, &s_mask, &s_inbin);
      __syncthreads();
      thr = s_prefix;
      if (shift == 32 && s_krem == s_inbin) {   // all keys of the boundary score stay
        thr |= 0xffffffffull;
        break;
      }
    }
    // keys <= thr, compacted in index order (in place when cached: every
    // thread reads its keys before any is written)
    constexpr int kPer = kGateSortMax / kSelThreads;
    unsigned long long mine[kPer];
    int cnt = 0;
    if (cached) {
      unsigned keep = 0;   // bit j: key tid * kPer + j stays
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = tid * kPer + j;
        mine[j] = i < T ? sk[i] : 0ull;
        if (i < T && mine[j] <= thr) keep |= 1u << j;
      }
      cnt = __popc(keep);
      int total;
      int pos = block_exclusive_scan(cnt, &total, sh_i);   // synchronises the reads
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        if (keep & (1u << j)) sk[pos++] = mine[j];
    } else {
      for (int i = tid; i < T; i += kSelThreads) {
        const unsigned long long key = ec_key(col, i);
        if (key <= thr) {
          const int pos = atomicAdd(&s_cnt, 1);
          if (pos < kGateSortMax) sk[pos] = key;
        }
      }
    }
  }
  __syncthreads();
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = k + tid; i < P; i += kSelThreads) sk[i] = ~0ull;
  __syncthreads();
  bitonic_sort_asc(sk, P);
  const size_t base = (size_t)e * a.C;
  for (int i = tid; i < a.C; i += kSelThreads) {
    int t = -1;
    float g = 0.f;
    if (i < k) {
      t = (int)(unsigned)(sk[i] & 0xffffffffull);
      g = __uint_as_float(~(unsigned)(sk[i] >> 32));
      atomicAdd(a.per_token + t, 1);
      if (a.tok_of_slot) {
        a.tok_of_slot[base + i] = t;
        a.slot_gate[base + i] = g;
      }
    }
    a.chosen_token[base + i] = t;
    a.chosen_gate[base + i] = g;
  }
  if (a.xbuf) {   // dispatch: one warp per kept row
    const uint32_t rb = (uint32_t)a.d * (uint32_t)a.elem_bytes;
    for (int i = warp; i < k; i += kSelThreads / 32) {
      const int t = (int)(unsigned)(sk[i] & 0xffffffffull);
      copy_row(static_cast<const char*>(a.x) + (size_t)t * rb,
               static_cast<char*>(a.xbuf) + (base + i) * rb, (int)rb, lane);
    }
  }
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s, bool pdl) {
  return launch_k(scan_kernel, dim3(a.hist2 ? 2 * a.N : a.N), dim3(kScanThreads), 0, s, pdl, a);
}

// Dynamic shared memory of the row-staging kernels: one row per warp when
// the rows are staged through TMA.
static size_t row_stage_smem(const AssignArgs& a, bool dispatch) {
  const size_t rb = (size_t)a.d * a.elem_bytes;
  const bool staged = (dispatch || (a.mode == SWITCH_MOE_TOKEN_ORDER && a.xbuf)) &&
                      rb <= kStageRowMax;
  return staged ? (size_t)kRowWarps * rb : 0;
}

cudaError_t launch_assign(const AssignArgs& a, const ScanArgs* finish, cudaStream_t s, bool pdl) {
  const size_t smem = row_stage_smem(a, false);
  cudaError_t err =
      cudaFuncSetAttribute(assign_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  ScanArgs sa{};
  if (finish) sa = *finish;
  const int grid = (a.T + kRowWarps - 1) / kRowWarps + (sa.defer_finish ? 1 : 0);
  return launch_k(assign_kernel, dim3(grid), dim3(kRowWarps * 32), smem, s, pdl, a, sa);
}

cudaError_t launch_dispatch(const AssignArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = row_stage_smem(a, true);
  cudaError_t err = cudaFuncSetAttribute(dispatch_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_k(dispatch_kernel, dim3((a.T + kRowWarps - 1) / kRowWarps), dim3(kRowWarps * 32),
                  smem, s, pdl, a);
}

cudaError_t launch_expert_select(const ExpertChoiceArgs& a, const ScanArgs& fin, cudaStream_t s,
                                 bool pdl) {
  const size_t smem = (size_t)kGateSortMax * sizeof(unsigned long long);
  cudaError_t err = cudaFuncSetAttribute(expert_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_k(expert_select_kernel, dim3(a.N + 1), dim3(kSelThreads), smem, s, pdl, a, fin);
}

cudaError_t launch_gate_select(const AssignArgs& a, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)kGateSortMax * sizeof(unsigned long long);
  cudaError_t err = cudaFuncSetAttribute(gate_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_k(gate_select_kernel, dim3(a.N), dim3(kSelThreads), smem, s, pdl, a);
}

}  // namespace smoe

namespace smoe {

cudaError_t launch_expand(const ExpandArgs& a, const ScanArgs& fin, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)(kExpandWarps + 1) * a.N * sizeof(int);
  cudaError_t err = cudaFuncSetAttribute(expand_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_k(expand_kernel, dim3(1), dim3(kExpandThreads), smem, s, pdl, a, fin);
}

cudaError_t launch_expand_dispatch(const ExpandArgs& a, cudaStream_t s, bool pdl) {
  const int grid = std::min((a.T + kRowWarps - 1) / kRowWarps, 4 * 148);   // 4 per SM
  return launch_k(expand_dispatch_kernel, dim3(grid), dim3(kRowWarps * 32), 0, s, pdl, a);
}

}  // namespace smoe
