// Expert FFN contractions for fp32 layers, in exact fp32 (FFMA).
//
// Tensor cores have no fp32 mode: TF32 keeps 10 mantissa bits and, with the
// weights read as stored (low bits ignored), moves y by about 0.5-1 % of
// rms(y) on the fp32 layer shape -- too close to the 1e-2 budget.  fp32
// layers therefore run this tiled FFMA kernel; bf16 layers use gemm_tc.cu.
//
// Same work decomposition and epilogue contract as the tensor-core path:
// a work tile is (expert, 32-token tile, 64-row weight tile);
//   epi 0: out0 = relu(D) (fp32), epi 1: out0 = D (fp32).
#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int BM = 64, BNT = kSimtTileN, BK = 32, NT = 256;

__global__ void __launch_bounds__(NT) gemm_simt_kernel(const float* __restrict__ A,
                                                       const float* __restrict__ B, GemmArgs g) {
  __shared__ __align__(16) float As[BK][BM + 4];
  __shared__ __align__(16) float Bs[BK][BNT + 4];
  grid_dep_wait();
  grid_dep_launch();
  const int n_entries = g.entries ? *g.n_entries : g.n_entries_dense;
  const int tile = blockIdx.x;
  if (tile >= n_entries * g.m_tiles) return;
  const int j = tile / g.m_tiles, mt = tile - j * g.m_tiles;
  int e, nt;
  if (g.entries) {
    const int2 en = g.entries[j];
    e = en.x;
    nt = en.y;
  } else {
    e = 0;
    nt = j;
  }
  const int kept = g.counts ? min(g.counts[e], g.cap) : g.rows_per_expert;
  const int nv = min(BNT, kept - nt * BNT);
  const int tid = threadIdx.x, tm = tid & 15, tn = tid >> 4;   // rows tm*4.., tokens tn*2..
  const float* Ae = A + (size_t)e * g.M * g.K;
  const float* Be = B + ((size_t)e * g.rows_per_expert + (size_t)nt * BNT) * g.K;
  float acc[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = 0; k0 < g.K; k0 += BK) {
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int idx = tid + rep * NT, r = idx >> 3, c4 = (idx & 7) * 4;
      const int m = mt * BM + r, k = k0 + c4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < g.M && k < g.K) v = *reinterpret_cast<const float4*>(Ae + (size_t)m * g.K + k);
      As[c4 + 0][r] = v.x; As[c4 + 1][r] = v.y; As[c4 + 2][r] = v.z; As[c4 + 3][r] = v.w;
    }
    {
      const int r = tid >> 3, c4 = (tid & 7) * 4, k = k0 + c4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < nv && k < g.K) v = *reinterpret_cast<const float4*>(Be + (size_t)r * g.K + k);
      Bs[c4 + 0][r] = v.x; Bs[c4 + 1][r] = v.y; Bs[c4 + 2][r] = v.z; Bs[c4 + 3][r] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < BK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&As[k][tm * 4]);
      const float2 b = *reinterpret_cast<const float2*>(&Bs[k][tn * 2]);
      acc[0][0] = fmaf(a.x, b.x, acc[0][0]); acc[0][1] = fmaf(a.x, b.y, acc[0][1]);
      acc[1][0] = fmaf(a.y, b.x, acc[1][0]); acc[1][1] = fmaf(a.y, b.y, acc[1][1]);
      acc[2][0] = fmaf(a.z, b.x, acc[2][0]); acc[2][1] = fmaf(a.z, b.y, acc[2][1]);
      acc[3][0] = fmaf(a.w, b.x, acc[3][0]); acc[3][1] = fmaf(a.w, b.y, acc[3][1]);
    }
    __syncthreads();
  }
  float* out = static_cast<float*>(g.out0);
  const size_t row0 = (size_t)e * g.rows_per_expert + (size_t)nt * BNT;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = mt * BM + tm * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int jn = 0; jn < 2; ++jn) {
      const int c = tn * 2 + jn;
      if (c < nv) {
        const float v = acc[i][jn];
        out[(row0 + c) * (size_t)g.ldo + m] = g.epi == 0 ? fmaxf(v, 0.f) : v;
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& g, const float* A, const float* B, cudaStream_t s,
                             bool pdl) {
  if (g.grid <= 0) return cudaSuccess;
  return launch_k(gemm_simt_kernel, dim3(g.grid), dim3(NT), 0, s, pdl, A, B, g);
}

}  // namespace smoe
