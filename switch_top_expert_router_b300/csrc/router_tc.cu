// Router logits on the tcgen05 tensor cores for bf16 layers, fused with the
// softmax / top-1 / gate / P-partial / histogram epilogue.
//
// Sources: "Top-1 路由 (Top-1 Routing)" (compassingai.com), core mechanism
// steps 1-2 (score = softmax(W_g x); expert_id = argmax; gate_value =
// score[expert_id]); Switch Transformer walk-through
// (personwebsite.pages.dev/moe-switch), selective-precision section: the
// router computes in float32 although activations are bf16.
//
// Exactness.  x is bf16.  The fp32 router weights are split once per call
// into three bf16 pieces, W_g = W_hi + W_mid + W_lo: each piece is the
// bf16 rounding of what the previous ones left, every residual is exact in
// fp32, and the three pieces carry about 24 significant bits (the pieces'
// sum equals W_g to within 2^-26 relative).  Every product of a bf16 x and a
// bf16 piece is exact in fp32, so three bf16 MMAs accumulating in fp32
// give fp32-router logits.  (Plain TF32 or one bf16 copy of W_g would move
// the logits by ~1e-4, far past the 1e-5 routing-margin rule.)
//
// Promotion.  The tensor core's fp32 accumulation loses precision over long
// chains (measured on B300: logit error std 1.4e-6 at d_model 768 and 2.5e-5
// at 5120 when all of K accumulates in TMEM, against 2.7e-7 / 1.8e-6 for
// sequential FFMA).  So each 64-wide K block (4 k-steps x 3 pieces = 12
// MMAs) accumulates into a fresh TMEM accumulator, and the epilogue warps
// add that block sum into an fp32 running sum -- in registers for up to 128
// experts, else in TMEM -- with exact fp32 additions, one per block.  Two block accumulators alternate so the MMAs of
// block k+1 overlap the promotion of block k (one when 3 x N columns do not
// fit in TMEM).
//
// CTA = 128 tokens (MMA M) x all experts (MMA N = N rounded up to 16,
// <= 256), K = d_model in 64-wide TMA stages:
//   warp 0     TMA: x tile [128 x 64] + the three W_g pieces [n x 64]
//   warp 1     TMEM allocator + MMA issuer (3 MMAs per 16-wide k step)
//   warps 2-5  promotion of every K block, then the epilogue: one thread
//              per token runs its N logits (staged in shared memory, or read
//              from TMEM) in increasing expert order -- the same operation
//              sequence as the FFMA router's epilogue, so both route
//              identical logits identically, bit for bit.
// Outputs per group of 32 tokens (one epilogue warp), the layout the scan
// expects: expert histogram, each token's rank among earlier same-expert
// tokens of the group, and the group's sum of probabilities per expert.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kXBytes = 128u * 128u;   // 128 tokens x 64 bf16
constexpr size_t kSmemLimit = 232448;
constexpr size_t kBarrierArea = 256;

__global__ void split_wg_kernel(const float* __restrict__ W_g, __nv_bfloat16* __restrict__ out,
                                int N, int n_pad, int d) {
  grid_dep_launch();   // first kernel of the layer: nothing before it is in flight
  const size_t total = (size_t)n_pad * d;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(idx / d);
    const float w = e < N ? W_g[idx] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);       // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);     // exact
    out[idx] = hi;
    out[total + idx] = mid;
    out[2 * total + idx] = __float2bfloat16_rn(r2);
  }
}

constexpr int kRegExperts = 128;   // experts whose running sums fit in registers

// Row stride (floats) of the finished logits staged in shared memory for the
// routing step: odd, so a warp reading one column of 32 rows, or 32
// consecutive columns of one row, touches 32 different banks.
constexpr int kEpiLd = kRegExperts + 1;
constexpr size_t kEpiBytes = (size_t)128 * kEpiLd * 4 + 128 * 4;   // logits + 1 / sums

// top-2: histogram and in-group ranks of one 32-token group's second
// choices e2 (-1 - lane past T), through this warp's histogram hs, which
// holds the first choices' histogram on entry (already stored).
__device__ __noinline__ void second_choice_hist(const RouterArgs& a, int* hs, int e2, bool valid,
                                                int lane, int t, int g) {
  const int N = a.N;
  __syncwarp();
  for (int i = lane; i < N; i += 32) hs[i] = 0;
  __syncwarp();
  const unsigned peers = __match_any_sync(0xffffffffu, e2);
  if (valid) {
    const unsigned lt = (1u << lane) - 1u;
    a.local_rank2[t] = __popc(peers & lt);
    if ((peers & lt) == 0) hs[e2] = __popc(peers);
  }
  __syncwarp();
  for (int i = lane; i < N; i += 32) a.hist2[(size_t)g * N + i] = hs[i];
}

// Routing of one epilogue warp's 32 tokens from their logits, staged in
// shared memory (row r = token t0 + r): expert id, gate, the group's
// per-expert probability sums and its histogram plus in-group ranks.  Each
// thread runs its token's row in increasing expert order, the same
// operation sequence as the FFMA router, so both route identical logits
// bit for bit.  Compact loops: this code runs once per launch, so its size,
// not its trip count, is what costs.
__device__ __noinline__ void route_group_smem(const RouterArgs& a, float* lg, float* invs,
                                              int* cnt_s, int q, int lane, int t0) {
  const int N = a.N, T = a.T;
  const int r = q * 32 + lane;
  const int t = t0 + r;
  const bool valid = t < T;
  float* row = lg + (size_t)r * kEpiLd;
  if (a.logits_out) {   // debug entry point: the logits only
    if (valid)
      for (int i = 0; i < N; ++i) a.logits_out[(size_t)t * N + i] = row[i];
    return;
  }
  float m = -INFINITY;
  int mi = 0;
  for (int i = 0; i < N; ++i) {
    const float v = row[i];
    if (v > m) {
      m = v;
      mi = i;
    }
  }
  int cand[kMaxCand];
  float cv[kMaxCand];
  if (a.n_cand > 1) topk_candidates([&](int i) { return row[i]; }, N, cand, cv);
  float s = 0.f;
  for (int i = 0; i < N; ++i) {
    const float e = expf(row[i] - m);
    row[i] = e;
    s += e;
  }
  const float inv = 1.0f / s;
  invs[r] = inv;
  if (valid) {
    a.expert_id[t] = mi;
    a.gate[t] = inv;   // exp(0) / s: the probability of the argmax
    for (int c = 0; c < a.n_cand && a.n_cand > 1; ++c) {
      a.cand[(size_t)t * kMaxCand + c] = cand[c];
      a.cand_p[(size_t)t * kMaxCand + c] = row[cand[c]] * inv;   // exp(l - m) / s
    }
  }
  __syncwarp();
  const int nvalid = min(32, T - (t0 + q * 32));
  if (nvalid <= 0) return;
  const int g = blockIdx.x * 4 + q;   // 32-token group
  // group sums of p = exp(l - m) / s per expert, tokens in order
  const float* rows = lg + (size_t)q * 32 * kEpiLd;
  float* pt = a.probs_t;   // expert choice: the probabilities, transposed
  for (int c = lane; c < N; c += 32) {
    float acc = 0.f;
    for (int rr = 0; rr < nvalid; ++rr) {
      const float pv = rows[(size_t)rr * kEpiLd + c] * invs[q * 32 + rr];
      acc += pv;
      if (pt) pt[(size_t)c * T + t0 + q * 32 + rr] = pv;
    }
    a.P_part[(size_t)g * N + c] = acc;
  }
  // histogram and rank among earlier same-expert tokens of the group
  const int e = valid ? mi : -1 - lane;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  int* hs = cnt_s + q * N;
  if (valid) {
    const unsigned lt = (1u << lane) - 1u;
    a.local_rank[t] = __popc(peers & lt);
    if ((peers & lt) == 0) hs[e] = __popc(peers);
  }
  __syncwarp();
  for (int i = lane; i < N; i += 32) a.hist[(size_t)g * N + i] = hs[i];
  if (a.hist2) second_choice_hist(a, hs, valid ? cand[1] : -1 - lane, valid, lane, t, g);
}

// Epilogue warps for N <= kRegExperts: promote every K block's TMEM sum
// into registers (running[i] += block[i], the same fp32 additions in the
// same order as the TMEM-resident variant), then route the token.
__device__ __forceinline__ void router_epilogue_regs(
    const RouterArgs& a, uint32_t taddr, int n_mma, int k_blocks, bool dbl, uint64_t* tfull,
    uint64_t* tempty, volatile int* abort_flag, int* status, uint8_t* tiles,
    const float* bias_s, int* cnt_s, int q, int lane, int t0, int t, bool valid) {
  const int nch = n_mma >> 4;   // 16-column chunks, <= 8
  float run[kRegExperts];
#pragma unroll
  for (int i = 0; i < kRegExperts; ++i) run[i] = 0.f;
  for (int kb = 0; kb < k_blocks; ++kb) {
    const int b = dbl ? (kb & 1) : 0;
    const uint32_t use = dbl ? (uint32_t)(kb >> 1) : (uint32_t)kb;
    const bool ready =
        mbar_wait(&tfull[b], use & 1u, abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
    if (!__all_sync(0xffffffffu, ready)) return;   // tcgen05.ld is warp-collective
    tc_fence_after();
    const uint32_t blk = taddr + (uint32_t)((1 + b) * n_mma);
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // 4 chunks (64 columns) in flight at a time
      uint32_t r[4][16];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (h * 4 + c < nch) tmem_ld_32x32b_x16_async(blk + (uint32_t)((h * 4 + c) * 16), r[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (h * 4 + c < nch) {
          tmem_wait_ld_regs(r[c]);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int i = (h * 4 + c) * 16 + j;
            run[i] = kb == 0 ? __uint_as_float(r[c][j]) : run[i] + __uint_as_float(r[c][j]);
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[b]);
  }
  if (a.part_out) {   // K split: this range's sums only; the FFMA kernel routes
    if (valid) {
      float* dst = a.part_out + ((size_t)blockIdx.y * a.T + t) * a.N;
#pragma unroll
      for (int i = 0; i < kRegExperts; ++i)
        if (i < a.N) dst[i] = run[i];
    }
    return;
  }
  // stage the finished logits (bias added) in the idle pipeline buffers
  float* lg = reinterpret_cast<float*>(tiles);
  float* row = lg + (size_t)(q * 32 + lane) * kEpiLd;
#pragma unroll
  for (int i = 0; i < kRegExperts; ++i)
    if (i < a.N) row[i] = run[i] + bias_s[i];
  __syncwarp();
  route_group_smem(a, lg, lg + (size_t)128 * kEpiLd, cnt_s, q, lane, t0);
}

// kRegs (N <= kRegExperts): each epilogue thread keeps its token's running
// sums in registers; otherwise they live in TMEM column block 0.
template <bool kRegs>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const RouterArgs a, int n_mma, int k_per, int k_total, int stages,
                     int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t w_bytes = (uint32_t)n_mma * 128u;
  const uint32_t stage_bytes = kXBytes + 3u * w_bytes;
  uint8_t* tiles = smem;
  const size_t tile_area = max((size_t)stages * stage_bytes, kEpiBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + tile_area);
  uint64_t* empty = full + stages;
  uint64_t* tfull = empty + stages;   // [2] block accumulator ready
  uint64_t* tempty = tfull + 2;       // [2] block accumulator promoted
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* bias_s = reinterpret_cast<float*>(tmem_slot + 4);          // [N]
  int* cnt_s = reinterpret_cast<int*>(bias_s + kMaxExpertsTc);      // [4][N] per-warp histograms

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N, T = a.T;
  const int t0 = blockIdx.x * 128;
  // K range of this CTA (blockIdx.y > 0 only when the router is split along K)
  const int kb0 = (int)blockIdx.y * k_per;
  const int k_blocks = min(k_per, k_total - kb0);
  // TMEM: running sum at column 0, block accumulators after it
  const bool dbl = 3 * n_mma <= 512;
  const int nacc = dbl ? 2 : 1;
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)((1 + nacc) * n_mma)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (blockIdx.x == 0 && a.ctrl) a.ctrl[0] = 0;   // done counter of the scan that follows
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  for (int i = threadIdx.x; i < N; i += kThreads) bias_s[i] = a.b_g ? a.b_g[i] : 0.f;
  for (int i = threadIdx.x; i < 4 * N; i += kThreads) cnt_s[i] = 0;
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x != 0) {   // thread 0, the producer, waits after its first x loads
    grid_dep_wait();
    grid_dep_launch();
  }

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_x = l2_policy_evict_first();
      const uint64_t pol_w = l2_policy_evict_last();   // every CTA reads all of W_g
      // x is the caller's input: its first stages load while the kernel
      // that splits W_g may still be running
      const int npre = min(stages, k_blocks);
      for (int kb = 0; kb < npre; ++kb) {
        mbar_arrive_expect_tx(&full[kb], stage_bytes);
        tma_load_2d(tiles + (size_t)kb * stage_bytes, &tmX, &full[kb], (kb0 + kb) * kTileK, t0,
                    pol_x);
      }
      grid_dep_wait();
      grid_dep_launch();
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      for (int kb = 0; kb < k_blocks; ++kb) {
        uint8_t* st = tiles + (size_t)stage * stage_bytes;
        const int kx = (kb0 + kb) * kTileK;
        if (kb >= npre) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status,
                         SWITCH_MOE_ERR_DEVICE_TIMEOUT))
            break;
          mbar_arrive_expect_tx(&full[stage], stage_bytes);
          tma_load_2d(st, &tmX, &full[stage], kx, t0, pol_x);
        }
        for (int pc = 0; pc < 3; ++pc)
          tma_load_2d(st + kXBytes + pc * w_bytes, &tmW, &full[stage], kx, pc * n_mma, pol_w);
        ++issued;
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      const uint32_t S = (uint32_t)stages;
      for (uint32_t s = 0; s < S && s < issued; ++s) {
        const uint32_t last = s + S * ((issued - 1u - s) / S);
        const unsigned long long t0ns = globaltimer_ns();
        while (!mbar_try_wait(&full[s], (last / S) & 1u)) {
          if (globaltimer_ns() - t0ns > kWaitTimeoutNs) {
            atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128u, (uint32_t)n_mma);
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = 0; kb < k_blocks; ++kb) {
        const int b = dbl ? (kb & 1) : 0;
        const uint32_t use = dbl ? (uint32_t)(kb >> 1) : (uint32_t)kb;   // earlier uses of b
        if (!mbar_wait(&tempty[b], (use & 1u) ^ 1u, abort_flag, status,
                       SWITCH_MOE_ERR_DEVICE_TIMEOUT))
          break;
        tc_fence_after();
        if (!mbar_wait(&full[stage], phase, abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)((1 + b) * n_mma);
        const uint32_t x_addr = smem_u32(tiles + (size_t)stage * stage_bytes);
        const uint32_t w_addr = x_addr + kXBytes;
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(x_addr + (uint32_t)k * 32u);
#pragma unroll
          for (int pc = 0; pc < 3; ++pc)
            mma_bf16_ss(d_tmem, ad, smem_desc_sw128(w_addr + pc * w_bytes + (uint32_t)k * 32u),
                        idesc, (k | pc) != 0 ? 1u : 0u);   // fresh sum per K block
        }
        mma_commit(&empty[stage]);
        mma_commit(&tfull[b]);
        if (++stage == stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit(drain);
      const unsigned long long t0ns = globaltimer_ns();
      while (!mbar_try_wait(drain, 0u)) {
        if (globaltimer_ns() - t0ns > kWaitTimeoutNs) {
          atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lanes / tokens 32q .. 32q + 31
    const int row = q * 32 + lane;
    const int t = t0 + row;
    const bool valid = t < T;
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);   // running sum
    if constexpr (kRegs) {
      router_epilogue_regs(a, taddr, n_mma, k_blocks, dbl, tfull, tempty, abort_flag, status,
                           tiles, bias_s, cnt_s, q, lane, t0, t, valid);
    } else {
    float v[16];
    bool ready = true;
    for (int kb = 0; kb < k_blocks && ready; ++kb) {
      const int b = dbl ? (kb & 1) : 0;
      const uint32_t use = dbl ? (uint32_t)(kb >> 1) : (uint32_t)kb;
      ready = mbar_wait(&tfull[b], use & 1u, abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
      if (!__all_sync(0xffffffffu, ready)) {   // leave together: tcgen05.ld is warp-collective
        ready = false;
        break;
      }
      tc_fence_after();
      const uint32_t blk = taddr + (uint32_t)((1 + b) * n_mma);
      for (int c0 = 0; c0 < N; c0 += 16) {
        tmem_ld_32x32b_x16(blk + (uint32_t)c0, v);
        if (kb > 0) {
          float r[16];
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, r);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = r[j] + v[j];
        }
        tmem_st_32x32b_x16(taddr + (uint32_t)c0, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
    if (ready) {
      tc_fence_after();
      // pass 1: max and first argmax, increasing expert order
      float m = -INFINITY;
      int mi = 0;
      for (int c0 = 0; c0 < N; c0 += 16) {
        tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = c0 + j;
          if (i < N) {
            const float l = v[j] + bias_s[i];
            if (l > m) { m = l; mi = i; }
          }
        }
      }
      // pass 2: sum of exp(l - m), sequential
      float s = 0.f;
      for (int c0 = 0; c0 < N; c0 += 16) {
        tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = c0 + j;
          if (i < N) s += expf((v[j] + bias_s[i]) - m);
        }
      }
      const float inv = 1.0f / s;
      const int g = blockIdx.x * 4 + q;                // 32-token group
      const bool group_ok = t0 + q * 32 < T;
      if (!a.logits_out && valid) {
        a.expert_id[t] = mi;
        a.gate[t] = inv;
      }
      int c2 = -1;   // second choice (top-2)
      if (!a.logits_out && a.n_cand > 1) {
        // Expanded Drop / top-2 candidates: one more pass over the TMEM row
        // with the insertion of topk_candidates
        int cand[kMaxCand];
        float cl[kMaxCand];
#pragma unroll
        for (int qq = 0; qq < kMaxCand; ++qq) {
          cand[qq] = -1;
          cl[qq] = 0.f;
        }
        for (int c0 = 0; c0 < N; c0 += 16) {
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int i = c0 + j;
            if (i >= N) continue;
            float nv = v[j] + bias_s[i];
            int ni = i;
            bool moved = false;
#pragma unroll
            for (int qq = 0; qq < kMaxCand; ++qq) {
              if (moved || cand[qq] < 0 || nv > cl[qq]) {
                const float tv = cl[qq];
                const int ti = cand[qq];
                cl[qq] = nv;
                cand[qq] = ni;
                nv = tv;
                ni = ti;
                moved = true;
              }
            }
          }
        }
        if (valid) {
          for (int r = 0; r < a.n_cand; ++r) {
            a.cand[(size_t)t * kMaxCand + r] = cand[r];
            a.cand_p[(size_t)t * kMaxCand + r] = expf(cl[r] - m) * inv;
          }
        }
        c2 = cand[1];
      }
      // pass 3, 32 experts at a time: probabilities through this warp's
      // [32][33] slice of the (now idle) pipeline buffers, then the group's
      // per-expert sums with the tokens in order (zeros past T change
      // nothing).  The debug entry point stores the logits instead.
      float* pw = reinterpret_cast<float*>(tiles) + (size_t)q * 32 * 33;
      for (int c0 = 0; c0 < N; c0 += 32) {
        float v2[16];
        tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
        tmem_ld_32x32b_x16(taddr + (uint32_t)c0 + 16u, v2);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = c0 + j;
          const float acc = j < 16 ? v[j] : v2[j - 16];
          if (i < N) {
            const float l = acc + bias_s[i];
            if (a.logits_out) {
              if (valid) a.logits_out[(size_t)t * N + i] = l;
            } else {
              pw[lane * 33 + j] = valid ? expf(l - m) * inv : 0.f;
            }
          }
        }
        __syncwarp();
        if (!a.logits_out && group_ok && c0 + lane < N) {
          float acc = 0.f;
          for (int r = 0; r < 32; ++r) {
            acc += pw[r * 33 + lane];
            if (a.probs_t && t0 + q * 32 + r < T)
              a.probs_t[(size_t)(c0 + lane) * T + t0 + q * 32 + r] = pw[r * 33 + lane];
          }
          a.P_part[(size_t)g * N + c0 + lane] = acc;
        }
        __syncwarp();
      }
      if (!a.logits_out && group_ok) {
        // histogram and rank among earlier same-expert tokens of the group
        const int e = valid ? mi : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int* hs = cnt_s + q * N;
        if (valid) {
          const unsigned lt = (1u << lane) - 1u;
          a.local_rank[t] = __popc(peers & lt);
          if ((peers & lt) == 0) hs[e] = __popc(peers);
        }
        __syncwarp();
        for (int i = lane; i < N; i += 32) a.hist[(size_t)g * N + i] = hs[i];
        if (a.hist2) second_choice_hist(a, hs, valid ? c2 : -1 - lane, valid, lane, t, g);
      }
    }
    }   // !kRegs
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int router_tc_n_mma(int N) { return (N + 15) / 16 * 16; }

int router_tc_stages(int N, int d) {
  const size_t stage = kXBytes + 3u * (size_t)router_tc_n_mma(N) * 128u;
  const size_t fixed = 1024 + kBarrierArea + (size_t)kMaxExpertsTc * 4 * 5;
  int st = (int)((kSmemLimit - fixed) / stage);
  const int kb = (d + kTileK - 1) / kTileK;
  if (st > kb) st = kb;
  if (st > 8) st = 8;
  return st < 1 ? 1 : st;   // one stage always holds the epilogue's 4 x 32 x 33 floats
}

size_t router_tc_smem_bytes(int N, int d) {
  const size_t stage = kXBytes + 3u * (size_t)router_tc_n_mma(N) * 128u;
  size_t area = (size_t)router_tc_stages(N, d) * stage;
  if (area < kEpiBytes) area = kEpiBytes;   // the routing step reuses the stage buffers
  return area + 1024 + kBarrierArea + (size_t)kMaxExpertsTc * 4 * 5;
}

cudaError_t launch_split_wg(const float* W_g, __nv_bfloat16* pieces, int N, int d,
                            cudaStream_t s) {
  const int n_pad = router_tc_n_mma(N);
  const size_t total = (size_t)n_pad * d;
  int grid = (int)((total + 255) / 256);
  if (grid > 1184) grid = 1184;
  split_wg_kernel<<<grid, 256, 0, s>>>(W_g, pieces, N, n_pad, d);
  return cudaGetLastError();
}

cudaError_t launch_router_tc(const RouterArgs& a, const CUtensorMap& tmX, const CUtensorMap& tmW,
                             int* status, cudaStream_t s, bool pdl, int ksplit) {
  const int n_mma = router_tc_n_mma(a.N);
  const int stages = router_tc_stages(a.N, a.d);
  const size_t smem = router_tc_smem_bytes(a.N, a.d);
  const bool regs = a.N <= kRegExperts;
  auto kern = regs ? router_tc_kernel<true> : router_tc_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (a.T + 127) / 128;
  const int k_total = (a.d + kTileK - 1) / kTileK;
  const int k_per = (k_total + ksplit - 1) / ksplit;
  return launch_k(kern, dim3(grid, ksplit), dim3(kThreads), smem, s, pdl, tmX, tmW, a, n_mma,
                  k_per, k_total, stages, status);
}

}  // namespace smoe
