// Combine: back to token order, gate scale, zero fill for dropped tokens,
// shared-expert add.
//
//   y[t] = sum over the token's kept choices r of g_tr * sum_s O_s[e_tr * C + slot_tr]
//          (+ S[t]); 0 when every choice was dropped
//   g_tr = gate_tr when gate_multiply, else 1; one choice for top-1, two for top-2
//   (the weighted merge of "Top-1 路由 (Top-1 Routing)", comparison section)
//
// Sources: "Top-1 路由 (Top-1 Routing)" (compassingai.com), core mechanism
// step 3 (Switch returns the chosen expert's output unscaled) against the
// Switch Transformer walk-through (personwebsite.pages.dev/moe-switch),
// Switch-layer section (the gate value multiplies the expert output, Eq. 2)
// -- hence the flag; the walk-through's expert-capacity section and
// "MoE 专家容量因子与 Token 丢弃" (wiblog.cn), overflow section: a dropped
// token gets no expert transform and continues through the residual, so
// the MoE branch is zero for it; "Which Routing Does Each MoE Model Use?"
// (MarkTechPost digest), routing table: the shared expert runs on every token.
//
// One warp per token and 512-wide chunk of d_model (blockIdx.y: long rows
// spread over more warps), 16-byte vectors (fp32 in and out).
#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kWarps = 8;
constexpr int kChunkV = 128;   // float4 per warp along d_model

__global__ void __launch_bounds__(kWarps * 32) combine_kernel(CombineArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= a.T) return;
  const int nv = a.d >> 2;
  float4* y = reinterpret_cast<float4*>(a.y + (size_t)t * a.d);
  const float4* S = a.S ? reinterpret_cast<const float4*>(a.S + (size_t)t * a.d) : nullptr;
  const float4* O0 = nullptr;   // the kept choices' expert outputs, in choice order
  const float4* O1 = nullptr;
  float g0 = 0.f, g1 = 0.f;
  for (int r = 0; r < a.topk; ++r) {
    const size_t i = (size_t)t * a.topk + r;
    const int s = a.slot[i];
    if (s < 0) continue;
    const float4* o = reinterpret_cast<const float4*>(a.O + ((size_t)a.expert_id[i] * a.C + s) * a.d);
    const float g = a.gate_multiply ? a.gate[i] : 1.0f;
    if (!O0) {
      O0 = o;
      g0 = g;
    } else {
      O1 = o;
      g1 = g;
    }
  }
  const size_t ss = a.split_stride >> 2;
  auto expert_out = [&](const float4* O, int v) {   // sum of the K-split partials
    float4 acc = __ldg(O + v);
    for (int k = 1; k < a.ksplit; ++k) {
      const float4 o = __ldg(O + k * ss + v);
      acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    }
    return acc;
  };
  const int v1 = min(nv, ((int)blockIdx.y + 1) * kChunkV);
  for (int v = (int)blockIdx.y * kChunkV + lane; v < v1; v += 32) {
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (O0) {
      const float4 acc = expert_out(O0, v);
      res = make_float4(g0 * acc.x, g0 * acc.y, g0 * acc.z, g0 * acc.w);
    }
    if (O1) {
      const float4 acc = expert_out(O1, v);
      res.x += g1 * acc.x; res.y += g1 * acc.y; res.z += g1 * acc.z; res.w += g1 * acc.w;
    }
    if (S) {
      const float4 sv = __ldg(S + v);
      res.x += sv.x; res.y += sv.y; res.z += sv.z; res.w += sv.w;
    }
    y[v] = res;
  }
}

// Expert choice without the fused combine: one warp per filled slot adds
// g * (sum of its K-split partials) into its token's row, and one warp per
// token adds the shared expert's row; y was zeroed by the selection.  A
// token may be taken by several experts, so the adds are atomic.
__global__ void __launch_bounds__(kWarps * 32) combine_slots_kernel(SlotCombineArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kWarps + warp;
  const long long n_slots = (long long)a.N * a.C;
  const int nv = a.d >> 2;
  if (item < n_slots) {
    if ((int)(item % a.C) >= a.kept) return;
    const int t = a.tok_of_slot[item];
    const float g = a.gate_multiply ? a.slot_gate[item] : 1.0f;
    const float4* O = reinterpret_cast<const float4*>(a.O + (size_t)item * a.d);
    const size_t ss = a.split_stride >> 2;
    float* y = a.y + (size_t)t * a.d;
    const int v1 = min(nv, ((int)blockIdx.y + 1) * kChunkV);
    for (int v = (int)blockIdx.y * kChunkV + lane; v < v1; v += 32) {
      float4 acc = __ldg(O + v);
      for (int k = 1; k < a.ksplit; ++k) {
        const float4 o = __ldg(O + k * ss + v);
        acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
      }
      atomicAdd(reinterpret_cast<float4*>(y) + v,
                make_float4(g * acc.x, g * acc.y, g * acc.z, g * acc.w));
    }
  } else if (a.S && item < n_slots + a.T) {
    const size_t t = (size_t)(item - n_slots);
    const float4* S = reinterpret_cast<const float4*>(a.S + t * a.d);
    float* y = a.y + t * a.d;
    const int v1 = min(nv, ((int)blockIdx.y + 1) * kChunkV);
    for (int v = (int)blockIdx.y * kChunkV + lane; v < v1; v += 32) {
      const float4 sv = __ldg(S + v);
      atomicAdd(reinterpret_cast<float4*>(y) + v, sv);
    }
  }
}

}  // namespace

cudaError_t launch_combine_slots(const SlotCombineArgs& a, cudaStream_t s, bool pdl) {
  const long long items = (long long)a.N * a.C + (a.S ? a.T : 0);
  const unsigned chunks = (unsigned)((a.d / 4 + kChunkV - 1) / kChunkV);
  return launch_k(combine_slots_kernel, dim3((unsigned)((items + kWarps - 1) / kWarps), chunks),
                  dim3(kWarps * 32), 0, s, pdl, a);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  const unsigned chunks = (unsigned)((a.d / 4 + kChunkV - 1) / kChunkV);
  return launch_k(combine_kernel, dim3((a.T + kWarps - 1) / kWarps, chunks), dim3(kWarps * 32), 0,
                  s, pdl, a);
}

}  // namespace smoe
