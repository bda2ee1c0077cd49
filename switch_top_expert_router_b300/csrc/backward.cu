// Backward of the top-1 layer: the gradients of <dy, y> + aux_coef * L_aux
// with respect to x, W_g, b_g, W1, W2 (and W1s, W2s), given the forward's
// routing (expert_id, gate, slot, expert_counts).
//
// Sources: Switch Transformer walk-through (personwebsite.pages.dev/
// moe-switch), load-balancing section (the auxiliary loss enters the
// training loss with a coefficient); "Top-1 路由 (Top-1 Routing)"
// (compassingai.com), core mechanism steps 1-3 (y = g * E(x), g = p_e) and
// load-balancing section (L_aux = N * sum_i f_i P_i).  The routing
// decisions (argmax, capacity, slots) are piecewise constant and pass no
// gradient; f_i (argmax counts) is constant, so dL_aux / dp[t, i] =
// N * f_i / T; the gate gets dy . E(x) when gate_multiply is set; ReLU'(0)
// is taken as 0.  Softmax backward: dl = p * (dp - sum_i p_i dp_i).
//
// Everything is fp32 (bf16 inputs are widened exactly) on FFMA: one
// strided batched GEMM kernel covers every contraction of the backward --
// over d_model, over d_ff, and over an expert's filled slots or the batch's
// tokens for the weight gradients -- by its strides, so no operand is ever
// transposed in memory.  The forward's intermediates (dispatched rows, the
// expert's hidden activation and output, the router probabilities) are
// recomputed from the inputs.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kTM = 128, kTN = 128, kTK = 8;   // output tile, K step
constexpr int kBThreads = 256;                  // 16 x 16 threads, 8 x 8 outputs each

__device__ __forceinline__ float ld_as_float(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld_as_float(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// C_b[m, n] (+)= sum_k A_b[m, k] * B_b[n, k] for batch b = blockIdx.z, with
// A_b[m, k] = A[b * a_b + m * a_m + k * a_k] (B likewise) and
// C_b[m, n] = C[b * c_b + m * c_m + n * c_n].  Per-batch counts (null: the
// full M, N, K) limit the rows m, n and the reduction k of batch b.  Each
// thread holds an 8 x 8 block of the 128 x 128 tile; the K step of 8 is
// staged in shared memory, loaded along each operand's contiguous axis.
template <typename TA, typename TB>
__global__ void __launch_bounds__(kBThreads, 2) bgemm_kernel(BGemmArgs g, const TA* __restrict__ A,
                                                          const TB* __restrict__ B) {
  __shared__ __align__(16) float as[kTK][kTM + 4];
  __shared__ __align__(16) float bs[kTK][kTN + 4];
  const int b = blockIdx.z;
  const int M = g.mcount ? min(__ldg(g.mcount + b), g.M) : g.M;
  const int N = g.ncount ? min(__ldg(g.ncount + b), g.N) : g.N;
  const int K = g.k_chunk ? min(g.k_chunk, g.K - b * g.k_chunk)
                         : (g.kcount ? min(__ldg(g.kcount + b), g.K) : g.K);
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  if (m0 >= M || n0 >= N) return;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const size_t ab = (size_t)b * g.a_b, bb = (size_t)b * g.b_b;
  const bool a_k_fast = g.a_k == 1, b_k_fast = g.b_k == 1;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  // the next K step's operands are loaded into registers while this one's
  // FMAs run (one shared-memory stage, one register stage).  Each thread's
  // element positions in the tile are fixed: their offsets are computed
  // once, and a K step only adds k0 times the K stride.
  constexpr int kRA = kTM * kTK / kBThreads, kRB = kTN * kTK / kBThreads;
  float ra[kRA], rb[kRB];
  size_t offa[kRA], offb[kRB];
  int kka[kRA], kkb[kRB];
#pragma unroll
  for (int r = 0; r < kRA; ++r) {
    const int i = tid + r * kBThreads;
    const int mm = a_k_fast ? i / kTK : i % kTM;
    kka[r] = a_k_fast ? i % kTK : i / kTM;
    const bool ok = m0 + mm < M;
    offa[r] = ok ? ab + (size_t)(m0 + mm) * g.a_m + (size_t)kka[r] * g.a_k : 0;
    if (!ok) kka[r] = 1 << 30;   // never below K: the element reads as 0
  }
#pragma unroll
  for (int r = 0; r < kRB; ++r) {
    const int i = tid + r * kBThreads;
    const int nn = b_k_fast ? i / kTK : i % kTN;
    kkb[r] = b_k_fast ? i % kTK : i / kTN;
    const bool ok = n0 + nn < N;
    offb[r] = ok ? bb + (size_t)(n0 + nn) * g.b_n + (size_t)kkb[r] * g.b_k : 0;
    if (!ok) kkb[r] = 1 << 30;
  }
  auto fetch = [&](int k0) {
    const size_t sa = (size_t)k0 * g.a_k, sb = (size_t)k0 * g.b_k;
#pragma unroll
    for (int r = 0; r < kRA; ++r) ra[r] = k0 + kka[r] < K ? ld_as_float(A, offa[r] + sa) : 0.f;
#pragma unroll
    for (int r = 0; r < kRB; ++r) rb[r] = k0 + kkb[r] < K ? ld_as_float(B, offb[r] + sb) : 0.f;
  };
  auto stash = [&]() {
#pragma unroll
    for (int r = 0; r < kRA; ++r) {
      const int i = tid + r * kBThreads;
      const int mm = a_k_fast ? i / kTK : i % kTM, kk = a_k_fast ? i % kTK : i / kTM;
      as[kk][mm] = ra[r];
    }
#pragma unroll
    for (int r = 0; r < kRB; ++r) {
      const int i = tid + r * kBThreads;
      const int nn = b_k_fast ? i / kTK : i % kTN, kk = b_k_fast ? i % kTK : i / kTN;
      bs[kk][nn] = rb[r];
    }
  };
  if (K > 0) fetch(0);
  for (int k0 = 0; k0 < K; k0 += kTK) {
    stash();
    __syncthreads();
    if (k0 + kTK < K) fetch(k0 + kTK);
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&as[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&as[kk][ty * 8 + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&bs[kk][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&bs[kk][tx * 8 + 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  const size_t cb = (size_t)b * g.c_b;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + ty * 8 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + tx * 8 + j;
      if (n >= N) continue;
      float* c = g.C + cb + (size_t)m * g.c_m + (size_t)n * g.c_n;
      *c = g.accumulate ? *c + acc[i][j] : acc[i][j];
    }
  }
}

// Per token t with a slot: Xg[e C + s] = x[t] (fp32), dO[e C + s] =
// (gate_multiply ? g_t : 1) dy[t], tok[e C + s] = t.  One warp per token.
template <typename TX>
__global__ void __launch_bounds__(256) bwd_gather_kernel(BwdArgs a, const TX* __restrict__ x) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.T) return;
  const int s = a.slot[t];
  if (s < 0) return;
  const size_t row = (size_t)a.expert_id[t] * a.C + s;
  const float g = a.gate_multiply ? a.gate[t] : 1.f;
  for (int j = lane; j < a.d; j += 32) {
    a.Xg[row * a.d + j] = ld_as_float(x, (size_t)t * a.d + j);
    a.dO[row * a.d + j] = g * a.dy[(size_t)t * a.d + j];
  }
  if (lane == 0) a.tok[row] = t;
}

// H = relu(Hpre) in place over rows [0, kept_e) of each expert's slots.
__global__ void bwd_relu_kernel(float* H, const int32_t* counts, int C, int F) {
  const int e = blockIdx.y;
  const int kept = counts ? min(counts[e], C) : C;
  const size_t n = (size_t)kept * F;
  float* h = H + (size_t)e * C * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    h[i] = fmaxf(h[i], 0.f);
}

// dH *= (H > 0): the ReLU's derivative (0 at 0).
__global__ void bwd_mask_kernel(float* dH, const float* H, const int32_t* counts, int C, int F) {
  const int e = blockIdx.y;
  const int kept = counts ? min(counts[e], C) : C;
  const size_t n = (size_t)kept * F, base = (size_t)e * C * F;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    if (!(H[base + i] > 0.f)) dH[base + i] = 0.f;
}

// Per kept slot: dx[tok] += dX[slot] (one slot per token: no two warps touch
// one row) and, with gate_multiply, dgate[tok] = dy[tok] . O[slot].
__global__ void __launch_bounds__(256) bwd_scatter_kernel(BwdArgs a) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.T) return;
  const int s = a.slot[t];
  float dg = 0.f;
  if (s >= 0) {
    const size_t row = (size_t)a.expert_id[t] * a.C + s;
    for (int j = lane; j < a.d; j += 32) {
      a.dx[(size_t)t * a.d + j] += a.dX[row * a.d + j];
      if (a.gate_multiply) dg += a.dy[(size_t)t * a.d + j] * a.O[row * a.d + j];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, off);
  }
  if (lane == 0) a.dgate[t] = dg;
}

// Router backward per token (one warp): p = softmax(l), dp_i = [i == e_t]
// dgate_t + aux_coef N f_i / T, dl = p (dp - sum_i p_i dp_i); l is
// overwritten by dl.
__global__ void __launch_bounds__(256) bwd_router_kernel(BwdArgs a) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.T) return;
  float* l = a.L + (size_t)t * a.N;
  if (a.b_g)
    for (int i = lane; i < a.N; i += 32) l[i] += a.b_g[i];
  __syncwarp();
  float m = -INFINITY;
  for (int i = lane; i < a.N; i += 32) m = fmaxf(m, l[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float s = 0.f;
  for (int i = lane; i < a.N; i += 32) s += expf(l[i] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  const float inv = 1.f / s;
  const int e = a.expert_id[t];
  const float dg = a.dgate[t];
  const float T = (float)a.T;
  float pdp = 0.f;
  for (int i = lane; i < a.N; i += 32) {
    const float p = expf(l[i] - m) * inv;
    const float dp = (i == e ? dg : 0.f) + a.aux_coef * (float)a.N * ((float)a.counts[i] / T) / T;
    pdp += p * dp;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) pdp += __shfl_xor_sync(0xffffffffu, pdp, off);
  __syncwarp();
  for (int i = lane; i < a.N; i += 32) {
    const float p = expf(l[i] - m) * inv;
    const float dp = (i == e ? dg : 0.f) + a.aux_coef * (float)a.N * ((float)a.counts[i] / T) / T;
    l[i] = p * (dp - pdp);
  }
}

// db_g[i] = sum_t dl[t, i]: one CTA per expert, a fixed-order block sum.
__global__ void __launch_bounds__(256) bwd_colsum_kernel(const float* dl, float* out, int T,
                                                         int N) {
  __shared__ float sh[256];
  const int i = blockIdx.x;
  float acc = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) acc += dl[(size_t)t * N + i];
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[i] = sh[0];
}

__global__ void bwd_sum_kernel(const float* __restrict__ parts, int n_parts, size_t n,
                               float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int p = 0; p < n_parts; ++p) acc += parts[(size_t)p * n + i];
    out[i] = acc;
  }
}

}  // namespace

cudaError_t launch_bwd_sum(const float* parts, int n_parts, size_t n, float* out,
                           cudaStream_t s) {
  const int grid = (int)std::min<size_t>((n + 255) / 256, 4 * 148);
  bwd_sum_kernel<<<grid, 256, 0, s>>>(parts, n_parts, n, out);
  return cudaGetLastError();
}

cudaError_t launch_bgemm(const BGemmArgs& g, const void* A, bool a_bf16, const void* B,
                         bool b_bf16, cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || g.batches <= 0) return cudaSuccess;
  const dim3 grid((g.N + kTN - 1) / kTN, (g.M + kTM - 1) / kTM, g.batches);
  if (a_bf16 && b_bf16)
    bgemm_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kBThreads, 0, s>>>(
        g, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B));
  else if (a_bf16)
    bgemm_kernel<__nv_bfloat16, float><<<grid, kBThreads, 0, s>>>(
        g, static_cast<const __nv_bfloat16*>(A), static_cast<const float*>(B));
  else if (b_bf16)
    bgemm_kernel<float, __nv_bfloat16><<<grid, kBThreads, 0, s>>>(
        g, static_cast<const float*>(A), static_cast<const __nv_bfloat16*>(B));
  else
    bgemm_kernel<float, float><<<grid, kBThreads, 0, s>>>(g, static_cast<const float*>(A),
                                                           static_cast<const float*>(B));
  return cudaGetLastError();
}

cudaError_t launch_bwd_gather(const BwdArgs& a, const void* x, bool x_bf16, cudaStream_t s) {
  const dim3 grid((a.T + 7) / 8);
  if (x_bf16)
    bwd_gather_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a,
                                                          static_cast<const __nv_bfloat16*>(x));
  else
    bwd_gather_kernel<float><<<grid, 256, 0, s>>>(a, static_cast<const float*>(x));
  return cudaGetLastError();
}

cudaError_t launch_bwd_relu(float* H, const int32_t* counts, int C, int F, int N, cudaStream_t s) {
  bwd_relu_kernel<<<dim3(64, N), 256, 0, s>>>(H, counts, C, F);
  return cudaGetLastError();
}

cudaError_t launch_bwd_mask(float* dH, const float* H, const int32_t* counts, int C, int F,
                            int batches, cudaStream_t s) {
  bwd_mask_kernel<<<dim3(64, batches), 256, 0, s>>>(dH, H, counts, C, F);
  return cudaGetLastError();
}

cudaError_t launch_bwd_scatter(const BwdArgs& a, cudaStream_t s) {
  bwd_scatter_kernel<<<(a.T + 7) / 8, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_router(const BwdArgs& a, cudaStream_t s) {
  bwd_router_kernel<<<(a.T + 7) / 8, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_colsum(const float* dl, float* out, int T, int N, cudaStream_t s) {
  bwd_colsum_kernel<<<N, 256, 0, s>>>(dl, out, T, N);
  return cudaGetLastError();
}

}  // namespace smoe
