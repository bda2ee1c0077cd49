// Combine: back to token order, gate scale, zero fill for dropped tokens,
// shared-expert add.
//
//   y[t] = (dropped ? 0 : g_t * sum_s O_s[e_t * C + slot_t]) + S[t]
//   g_t  = gate_t when gate_multiply, else 1
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
// One warp per token, 16-byte vectors along d_model (fp32 in and out).
#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) combine_kernel(CombineArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + warp;
  if (t >= a.T) return;
  const int s = a.slot[t];
  const int nv = a.d >> 2;
  float4* y = reinterpret_cast<float4*>(a.y + (size_t)t * a.d);
  const float4* S = a.S ? reinterpret_cast<const float4*>(a.S + (size_t)t * a.d) : nullptr;
  if (s < 0) {
    for (int v = lane; v < nv; v += 32) y[v] = S ? __ldg(S + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int e = a.expert_id[t];
  const float g = a.gate_multiply ? a.gate[t] : 1.0f;
  const float4* O = reinterpret_cast<const float4*>(a.O + ((size_t)e * a.C + s) * a.d);
  const size_t ss = a.split_stride >> 2;
  for (int v = lane; v < nv; v += 32) {
    float4 acc = __ldg(O + v);
    for (int k = 1; k < a.ksplit; ++k) {
      const float4 o = __ldg(O + k * ss + v);
      acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    }
    acc.x *= g; acc.y *= g; acc.z *= g; acc.w *= g;
    if (S) {
      const float4 sv = __ldg(S + v);
      acc.x += sv.x; acc.y += sv.y; acc.z += sv.z; acc.w += sv.w;
    }
    y[v] = acc;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s, bool pdl) {
  return launch_k(combine_kernel, dim3((a.T + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, s, pdl,
                  a);
}

}  // namespace smoe
