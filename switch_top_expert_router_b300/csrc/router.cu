// Router: fp32 logits l = W_g x (+ b_g), softmax over the N experts, top-1
// argmax (lowest index on ties) and gate, fused with the per-CTA partial
// sums of the probabilities (for P_i of the auxiliary loss) and the per-CTA
// expert histogram plus in-CTA rank (for token-order slot assignment).
//
// Sources: "Top-1 路由 (Top-1 Routing)" (compassingai.com), core mechanism
// steps 1-2 (score = softmax(W_g x), expert_id = argmax, gate_value =
// score[expert_id]) and load-balancing section (P_i = mean probability);
// Switch Transformer walk-through (personwebsite.pages.dev/moe-switch),
// selective-precision section: the router runs in float32 even when the
// layer's activations are bf16.
//
// One CTA routes kRouterTM = 32 tokens with 256 threads.  The logits GEMM
// runs in expert chunks of 128 on FFMA; each thread owns a 4-token x
// 4-expert register tile.  The logits of the CTA's tokens stay in shared
// memory for the softmax and never touch HBM.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int TM = kRouterTM;
constexpr int EC = 128;   // experts per GEMM chunk
constexpr int KT = 32;    // K per shared-memory stage
constexpr int NTHREADS = 256;

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  // 4 bf16 = 8 bytes; rows are 16-byte aligned and the offset is a multiple of 4 elements
  uint2 u = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// logits of tokens [t0, t0 + TM) into lg[TM][ldl] (rows past T are zero).
template <typename XT>
__device__ void logits_tile(const XT* __restrict__ x, const float* __restrict__ W_g,
                            const float* __restrict__ b_g, int T, int d, int N, int t0,
                            float* lg, int ldl, float* xs, float* ws) {
  const int tid = threadIdx.x;
  const int ty = tid >> 5;   // 4 tokens: ty*4 .. ty*4+3
  const int tx = tid & 31;   // 4 experts: tx*4 .. tx*4+3 within the chunk
  for (int ec = 0; ec < N; ec += EC) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < d; k0 += KT) {
      {  // x tile: 32 tokens x 32 k -> xs[k][token]
        int r = tid >> 3, c4 = (tid & 7) * 4;
        int t = t0 + r, k = k0 + c4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T && k < d) v = load4(x + (size_t)t * d + k);  // d % 8 == 0: all 4 in range
        xs[(c4 + 0) * (TM + 4) + r] = v.x;
        xs[(c4 + 1) * (TM + 4) + r] = v.y;
        xs[(c4 + 2) * (TM + 4) + r] = v.z;
        xs[(c4 + 3) * (TM + 4) + r] = v.w;
      }
#pragma unroll
      for (int rep = 0; rep < 4; ++rep) {  // W tile: 128 experts x 32 k -> ws[k][expert]
        int r = rep * 32 + (tid >> 3), c4 = (tid & 7) * 4;
        int e = ec + r, k = k0 + c4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < N && k < d) v = load4(W_g + (size_t)e * d + k);
        ws[(c4 + 0) * (EC + 4) + r] = v.x;
        ws[(c4 + 1) * (EC + 4) + r] = v.y;
        ws[(c4 + 2) * (EC + 4) + r] = v.z;
        ws[(c4 + 3) * (EC + 4) + r] = v.w;
      }
      __syncthreads();
#pragma unroll 8
      for (int k = 0; k < KT; ++k) {
        float4 xv = *reinterpret_cast<const float4*>(xs + k * (TM + 4) + ty * 4);
        float4 wv = *reinterpret_cast<const float4*>(ws + k * (EC + 4) + tx * 4);
        const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
        const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wa[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = ec + tx * 4 + j;
      if (e < N) {
        float b = b_g ? b_g[e] : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) lg[(ty * 4 + i) * ldl + e] = acc[i][j] + b;
      }
    }
  }
  __syncthreads();
}

// Softmax / argmax / gate / P partials / histogram / in-CTA rank on lg (and
// with top-2 the same histogram and ranks of the second choices).
// One thread per token runs the row in increasing expert order (the same
// operation sequence as the tensor-core router's epilogue, so both give
// bit-identical results on identical logits):
//   m = max_i l_i, e = first i with l_i == m (lowest index wins ties),
//   s = sum_i exp(l_i - m) (sequential), gate = 1 / s, p_i = exp(l_i - m) / s.
__device__ void route_tile(float* lg, int ldl, int T, int N, int t0, int cta,
                           const RouterArgs& a, int* es, int* es2, int* hs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < TM && t0 + tid < T) {
    const int t = t0 + tid;
    float* row = lg + tid * ldl;
    float m = -INFINITY;
    int mi = 0;   // stays 0 only if every logit is NaN: keeps the index in range
    for (int i = 0; i < N; ++i) {
      const float v = row[i];
      if (v > m) { m = v; mi = i; }
    }
    float s = 0.f;
    for (int i = 0; i < N; ++i) s += expf(row[i] - m);
    const float inv = 1.0f / s;
    int cand[kMaxCand];
    float cv[kMaxCand];
    if (a.n_cand > 1) topk_candidates([&](int i) { return row[i]; }, N, cand, cv);
    for (int i = 0; i < N; ++i) row[i] = expf(row[i] - m) * inv;   // probabilities
    a.expert_id[t] = mi;
    a.gate[t] = inv;    // score of the argmax: exp(0) / s
    es[tid] = mi;
    if (a.hist2) es2[tid] = cand[1];
    for (int r = 0; r < a.n_cand && a.n_cand > 1; ++r) {
      a.cand[(size_t)t * kMaxCand + r] = cand[r];
      a.cand_p[(size_t)t * kMaxCand + r] = row[cand[r]];
    }
  }
  for (int i = tid; i < N; i += NTHREADS) hs[i] = 0;
  __syncthreads();
  // P partial of this CTA: fixed token order, so the result is reproducible
  const int nt = min(TM, T - t0);
  for (int i = tid; i < N; i += NTHREADS) {
    float acc = 0.f;
    for (int r = 0; r < nt; ++r) {
      acc += lg[r * ldl + i];
      if (a.probs_t) a.probs_t[(size_t)i * T + t0 + r] = lg[r * ldl + i];
    }
    a.P_part[(size_t)cta * N + i] = acc;
  }
  // histogram + rank among earlier same-expert tokens of this CTA (TM == 32)
  if (warp == 0) {
    const bool valid = lane < nt;
    const int e = valid ? es[lane] : -1 - lane;   // invalid lanes never match a real expert
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const unsigned lt = (1u << lane) - 1u;
      a.local_rank[t0 + lane] = __popc(peers & lt);
      if ((peers & lt) == 0) hs[e] = __popc(peers);   // lowest lane of the group
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += NTHREADS) a.hist[(size_t)cta * N + i] = hs[i];
  if (!a.hist2) return;
  // top-2: the same for every token's second choice
  __syncthreads();
  for (int i = tid; i < N; i += NTHREADS) hs[i] = 0;
  __syncthreads();
  if (warp == 0) {
    const bool valid = lane < nt;
    const int e = valid ? es2[lane] : -1 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const unsigned lt = (1u << lane) - 1u;
      a.local_rank2[t0 + lane] = __popc(peers & lt);
      if ((peers & lt) == 0) hs[e] = __popc(peers);
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += NTHREADS) a.hist2[(size_t)cta * N + i] = hs[i];
}

template <typename XT>
__global__ void __launch_bounds__(NTHREADS) router_kernel(RouterArgs a) {
  extern __shared__ float4 smem_f4[];
  grid_dep_wait();
  grid_dep_launch();
  float* smem = reinterpret_cast<float*>(smem_f4);
  const int ldl = a.N + 1;
  float* lg = smem;                                  // [TM][N + 1]
  float* xs = lg + ((TM * ldl + 3) & ~3);            // [KT][TM + 4]
  float* ws = xs + KT * (TM + 4);                    // [KT][EC + 4]
  int* es = reinterpret_cast<int*>(ws + KT * (EC + 4));  // [TM]
  int* es2 = es + TM;                                // [TM] second choices (top-2)
  int* hs = es2 + TM;                                // [N]
  const int t0 = blockIdx.x * TM;
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.ctrl) {
    a.ctrl[0] = 0;   // done counter of the scan kernel that follows
  }
  if (a.parts_in) {   // K-split tensor-core logits: the parts in order, then the bias
    for (int idx = threadIdx.x; idx < TM * a.N; idx += NTHREADS) {
      const int r = idx / a.N, i = idx - r * a.N;
      float v = 0.f;
      if (t0 + r < a.T) {
        for (int p = 0; p < a.n_parts; ++p) v += a.parts_in[((size_t)p * a.T + t0 + r) * a.N + i];
        if (a.b_g) v += a.b_g[i];
      }
      lg[r * ldl + i] = v;
    }
    __syncthreads();
  } else if (a.logits_in) {
    for (int idx = threadIdx.x; idx < TM * a.N; idx += NTHREADS) {
      int r = idx / a.N, i = idx - r * a.N;
      lg[r * ldl + i] = (t0 + r < a.T) ? a.logits_in[(size_t)(t0 + r) * a.N + i] : 0.f;
    }
    __syncthreads();
  } else {
    logits_tile<XT>(reinterpret_cast<const XT*>(a.x), a.W_g, a.b_g, a.T, a.d, a.N, t0, lg,
                    ldl, xs, ws);
  }
  if (a.logits_out) {
    for (int idx = threadIdx.x; idx < TM * a.N; idx += NTHREADS) {
      int r = idx / a.N, i = idx - r * a.N;
      if (t0 + r < a.T) a.logits_out[(size_t)(t0 + r) * a.N + i] = lg[r * ldl + i];
    }
    return;
  }
  route_tile(lg, ldl, a.T, a.N, t0, blockIdx.x, a, es, es2, hs);
}

size_t router_smem_bytes(int N) {
  size_t ldl = (size_t)N + 1;
  size_t f = ((TM * ldl + 3) & ~(size_t)3) + KT * (TM + 4) + KT * (EC + 4);
  return f * sizeof(float) + (2 * TM + (size_t)N) * sizeof(int);
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const int R = (a.T + TM - 1) / TM;
  const size_t smem = router_smem_bytes(a.N);
  cudaError_t err;
  if (a.x_is_bf16) {
    err = cudaFuncSetAttribute(router_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_kernel<__nv_bfloat16><<<R, NTHREADS, smem, s>>>(a);
  } else {
    err = cudaFuncSetAttribute(router_kernel<float>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_kernel<float><<<R, NTHREADS, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace smoe
