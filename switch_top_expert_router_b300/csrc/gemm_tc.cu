// Expert FFN contractions on the tcgen05 tensor cores (bf16 x bf16 -> fp32).
//
// The expert FFN is a two-layer bias-free MLP, about 2 * d_model * d_ff
// weights per expert ("Top-1 路由 (Top-1 Routing)", compassingai.com,
// key-parameter section); the per-expert [N, C, d_model] buffer gives the
// grouped GEMM a static shape ("MoE 专家容量因子与 Token 丢弃", wiblog.cn,
// section on where capacity comes from).  Only filled slots are computed.
//
// Orientation ("swap AB"): expert weights are the 128-row A operand (MMA M),
// the expert's tokens are the B operand (MMA N = token tile, 16..256), K is
// the contraction.  Both operands are K-major and arrive by TMA with the
// 128-byte swizzle, 64 bf16 (128 bytes) of K per pipeline stage.
//   GEMM1: H^T[f, c] = W1[e, f, :] . X[e, c, :]     -> relu -> H (bf16 hi + lo)
//   GEMM2: O^T[j, c] = W2[e, j, :] . (H_hi + H_lo)[e, c, :]   (two MMAs / k-step)
// H is stored as an unevaluated sum of two bf16 values so the second layer
// sees H with ~16 significant bits (a single bf16 rounding of H moves y by
// more than the 1e-2 * rms(y) budget at these sizes).
//
// Second layer of the routed experts: the epilogue is also the combine step
// -- each filled slot's row goes straight to its token's row of y, scaled by
// the gate when gate_multiply is set ("Top-1 路由 (Top-1 Routing)", core
// mechanism step 3, against the Switch Transformer walk-through's Switch
// layer, Eq. 2), so the expert outputs never round-trip through HBM.
//
// Tail split: tiles are handed out round-robin, so when the last wave is
// less than half full most SMs would idle while a few stream whole weight
// tiles.  Those last tiles are cut along K into equal pieces run by the idle
// CTAs; each piece stores its fp32 partial, and for every 32-row slice the
// last piece to finish (an atomic counter) adds the partials in piece order
// -- deterministic, whatever the finishing order -- and applies the epilogue.
//
// CTA = 6 warps, persistent over a static round-robin of work units
// (expert, token tile, 128-row weight tile, K range):
//   warp 0      TMA producer (one lane) into a `stages`-deep shared ring
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  epilogue: TMEM -> registers -> global, 32 TMEM lanes each
// Four TMEM accumulators (two for token tiles over 128) let the epilogue of
// tile i lag the MMAs of the following tiles.  Every wait is bounded; on a timeout the CTA records
// SWITCH_MOE_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and
// returns.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kABytes = kTileM * 128;     // 16 KB per stage
constexpr size_t kSmemLimit = 232448;          // opt-in dynamic shared memory per block
constexpr size_t kBarrierArea = 512;
constexpr int kMaxPieces = 4;          // K pieces per split tile (one round of partial loads)
constexpr int kMaxAcc = 4;             // TMEM accumulators in flight
constexpr int kMinPieceKBlocks = 4;    // 256 of K at least per piece

__device__ __forceinline__ void decode_tile(const GemmArgs& g, int tile, int& e, int& nt,
                                            int& mt, int& ks, int& nv) {
  const int per_entry = g.m_tiles * g.ksplit;
  const int j = tile / per_entry;
  const int rem = tile - j * per_entry;
  mt = rem / g.ksplit;
  ks = rem - mt * g.ksplit;
  if (g.entries) {
    const int2 en = g.entries[j];
    e = en.x;
    nt = en.y;
  } else {
    e = 0;
    nt = j;
  }
  const int kept = g.counts ? min(g.counts[e], g.cap) : g.rows_per_expert;
  nv = min(g.BN, kept - nt * g.BN);
}

// Tail split plan for `total` tiles over the grid: tiles [0, full) run whole,
// the remaining total - full tiles run as `pieces` K pieces each.
__device__ __forceinline__ void split_plan(const GemmArgs& g, int total, int& full,
                                           int& pieces) {
  full = total;
  pieces = 1;
  if (!g.part || g.ksplit != 1) return;
  const int grid = (int)gridDim.x;
  const int rem = total % grid;
  if (rem == 0 || 2 * rem > grid) return;
  int p = grid / rem;
  p = min(p, g.k_blocks / kMinPieceKBlocks);
  p = min(p, kMaxPieces);
  if (p < 2 || rem * p > g.part_units) return;
  full = total - rem;
  pieces = p;
}

struct Work {
  int e, nt, mt, ks, nv;
  int kb0, nkb;   // K blocks [kb0, kb0 + nkb)
  int unit;       // index of the piece among all split pieces, -1: whole tile
  int sidx;       // index of the split tile
  int pieces;
};

__device__ __forceinline__ void decode_work(const GemmArgs& g, int u, int full, int pieces,
                                            Work& w) {
  int tile = u;
  w.unit = -1;
  w.sidx = 0;
  w.pieces = pieces;
  int piece = 0;
  if (u >= full) {
    w.unit = u - full;
    w.sidx = w.unit / pieces;
    piece = w.unit - w.sidx * pieces;
    tile = full + w.sidx;
  }
  decode_tile(g, tile, w.e, w.nt, w.mt, w.ks, w.nv);
  if (w.unit < 0) {
    w.kb0 = w.ks * g.k_blocks;
    w.nkb = g.k_blocks;
  } else {
    w.kb0 = piece * g.k_blocks / pieces;
    w.nkb = (piece + 1) * g.k_blocks / pieces - w.kb0;
  }
}

// Bounded wait that ignores the abort flag: used at teardown to let copies
// and MMAs that are already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
  unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 0; it < kWaitMaxIters; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 31u) == 31u && globaltimer_ns() - t0 > kWaitTimeoutNs) break;
  }
  atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
}

// kEpi: the epilogue (GemmArgs::epi), fixed at compile time so each variant
// carries only its own store path; 3 is the combine with several slots per
// token (top-2, expert choice): gates per slot, atomic adds into y.
template <int kEpi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t b_bytes = (uint32_t)g.BN * 128u;
  const uint32_t stage_bytes = kABytes + (uint32_t)g.num_b * b_bytes;
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)g.stages * stage_bytes);
  uint64_t* empty = full + g.stages;
  uint64_t* tfull = empty + g.stages;   // [kMaxAcc] accumulator ready for the epilogue
  uint64_t* tempty = tfull + kMaxAcc;   // [kMaxAcc] accumulator drained by the epilogue
  uint64_t* drain = tempty + kMaxAcc;   // [1] MMA drain at teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // all 512 TMEM columns: four accumulators of 128 columns, or two of 256
  const uint32_t acc_stride = g.BN <= 128 ? 128u : 256u;
  const uint32_t n_acc = 512u / acc_stride;
  const uint32_t tmem_cols = 512u;
  int* status = g.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    if (g.num_b == 2) prefetch_tensormap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the work list and the B operand come from the kernel before this one
  grid_dep_wait();
  grid_dep_launch();

  const int n_entries = g.entries ? *g.n_entries : g.n_entries_dense;
  const int total = n_entries * g.m_tiles * g.ksplit;
  int full_tiles, pieces;
  split_plan(g, total, full_tiles, pieces);
  const int n_units = full_tiles + (total - full_tiles) * pieces;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_a = l2_policy_evict_first();   // weights: streamed once
      const uint64_t pol_b = l2_policy_evict_last();    // tokens: reused by every weight tile
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        Work w;
        decode_work(g, u, full_tiles, pieces, w);
        const int ya = w.e * g.M + w.mt * kTileM;
        const int yb = w.e * g.rows_per_expert + w.nt * g.BN;
        for (int kb = 0; kb < w.nkb; ++kb) {
          uint8_t* st = tiles + (size_t)stage * stage_bytes;
          const int kx = (w.kb0 + kb) * kTileK;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status,
                         SWITCH_MOE_ERR_DEVICE_TIMEOUT)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], stage_bytes);
          tma_load_2d(st, &tmA, &full[stage], kx, ya, pol_a);
          tma_load_2d(st + kABytes, &tmB0, &full[stage], kx, yb, pol_b);
          if (g.num_b == 2) tma_load_2d(st + kABytes + b_bytes, &tmB1, &full[stage], kx, yb, pol_b);
          ++issued;
          if (++stage == g.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every copy this CTA started land before it exits.
      const uint32_t S = (uint32_t)g.stages;
      for (uint32_t s = 0; s < S && s < issued; ++s) {
        const uint32_t last = s + S * ((issued - 1u - s) / S);   // latest issue on stage s
        drain_wait(&full[s], (last / S) & 1u, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0, it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++it) {
        Work w;
        decode_work(g, u, full_tiles, pieces, w);
        const uint32_t acc = it % n_acc, acc_par = (it / n_acc) & 1u;
        if (!mbar_wait(&tempty[acc], acc_par ^ 1u, abort_flag, status,
                       SWITCH_MOE_ERR_DEVICE_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_stride;
        const uint32_t n_mma = ((uint32_t)w.nv + 15u) & ~15u;
        const uint32_t idesc = idesc_bf16_f32(128u, n_mma);
        for (int kb = 0; kb < w.nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, status,
                         SWITCH_MOE_ERR_DEVICE_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + (size_t)stage * stage_bytes);
          const uint32_t b0_addr = a_addr + kABytes;
          const uint32_t b1_addr = b0_addr + b_bytes;
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {   // 16 bf16 = 32 bytes of K per MMA
            const uint64_t ad = smem_desc_sw128(a_addr + (uint32_t)k * 32u);
            mma_bf16_ss(d_tmem, ad, smem_desc_sw128(b0_addr + (uint32_t)k * 32u), idesc,
                        (kb | k) != 0 ? 1u : 0u);
            if (g.num_b == 2)
              mma_bf16_ss(d_tmem, ad, smem_desc_sw128(b1_addr + (uint32_t)k * 32u), idesc, 1u);
          }
          mma_commit(&empty[stage]);   // frees the stage once these MMAs have read it
          if (++stage == g.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);       // accumulator complete
      }
      mma_commit(drain);
      drain_wait(drain, 0u, status);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;   // TMEM lanes 32q .. 32q + 31 belong to this warp
    const unsigned kAll = 0xffffffffu;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
      Work w;
      decode_work(g, u, full_tiles, pieces, w);
      const uint32_t acc = it % n_acc, acc_par = (it / n_acc) & 1u;
      const int row = w.mt * kTileM + q * 32 + lane;   // weight row = output column
      const bool row_ok = row < g.M;
      const size_t out_row0 = (size_t)w.e * g.rows_per_expert + (size_t)w.nt * g.BN;
      // combine: token and gate of columns c .. c + 31, one column per lane
      auto tok_gate = [&](int c, int& tk, float& gv) {
        tk = 0;
        gv = 1.f;
        if (c + lane < w.nv) {
          tk = g.tok_of_slot[out_row0 + (size_t)(c + lane)];
          if (g.gate_multiply)   // several slots per token: the gate belongs to the slot
            gv = kEpi == 3 ? g.slot_gate[out_row0 + (size_t)(c + lane)] : g.gate[tk];
        }
      };
      int tk32 = 0;
      float gv32 = 1.f;
      if (kEpi >= 2 && w.unit < 0) tok_gate(0, tk32, gv32);   // overlaps the wait below
      // tcgen05.ld below is warp-collective: leave the loop together or not at all
      const bool ready =
          mbar_wait(&tfull[acc], acc_par, abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
      if (!__all_sync(kAll, ready)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * acc_stride;

      const size_t tile_elems = (size_t)kTileM * (size_t)g.BN;
      bool from_tmem = true;   // else: the sum of a split tile's parked partials
      const float* p0 = nullptr;
      if (w.unit >= 0) {
        // one K piece of a split tile: park the partial, [column][128 rows]
        float* mine = g.part + (size_t)w.unit * tile_elems + q * 32 + lane;
        for (int c0 = 0; c0 < w.nv; c0 += 16) {
          float v[16];
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < w.nv) mine[(size_t)(c0 + j) * kTileM] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          int32_t* cnt = g.split_cnt + w.sidx * 4 + q;
          last = atomicAdd(cnt, 1) == w.pieces - 1;
          if (last) *cnt = 0;   // every piece has arrived: reset for the next launch
        }
        if (!__shfl_sync(kAll, last, 0)) continue;
        __threadfence();
        from_tmem = false;
        p0 = g.part + (size_t)w.sidx * w.pieces * tile_elems + q * 32 + lane;
        if (kEpi >= 2) tok_gate(0, tk32, gv32);
      }
      // 16 columns c0 .. c0 + 15 of this thread's row into v
      auto fetch16 = [&](int c0, float (&v)[16]) {
        if (from_tmem) {
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
          return;
        }
        // every piece's loads in flight at once, then the sum in piece order
        float t[kMaxPieces][16];
#pragma unroll
        for (int i = 0; i < kMaxPieces; ++i) {
          const float* src = p0 + (size_t)i * tile_elems + (size_t)c0 * kTileM;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            t[i][j] = (i < w.pieces && c0 + j < w.nv) ? __ldcg(src + j * kTileM) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = t[0][j];
#pragma unroll
        for (int i = 1; i < kMaxPieces; ++i) {
          if (i < w.pieces) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = v[j] + t[i][j];
          }
        }
      };

      if constexpr (kEpi >= 2) {
        // combine: y[token] = g_token * D (+ y[token]), 32 columns per step
        float* y = static_cast<float*>(g.out0);
        for (int c0 = 0; c0 < w.nv; c0 += 32) {
          if (c0 > 0) tok_gate(c0, tk32, gv32);
          float v[2][16];
          fetch16(c0, v[0]);
          fetch16(c0 + 16, v[1]);
          if constexpr (kEpi == 3) {
            add_block_v4(v, tk32, gv32, y, g.ldo, w.mt * kTileM + q * 32, g.M, c0, w.nv, lane);
            continue;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tj = __shfl_sync(kAll, tk32, j);
            const float gj = __shfl_sync(kAll, gv32, j);
            if (row_ok && c0 + j < w.nv) {
              float* dst = y + (size_t)tj * (size_t)g.ldo + row;
              const float val = gj * v[j >> 4][j & 15];
              if constexpr (kEpi == 3) {
                atomicAdd(dst, val);   // several slots add into one row
              } else {
                *dst = g.y_acc ? *dst + val : val;
              }
            }
          }
        }
      } else {
        for (int c0 = 0; c0 < w.nv; c0 += 16) {
          float v[16];
          fetch16(c0, v);
          if (!row_ok) continue;
          if constexpr (kEpi == 0) {
            // relu, then H as an unevaluated bf16 pair hi + lo
            __nv_bfloat16* hi = static_cast<__nv_bfloat16*>(g.out0);
            __nv_bfloat16* lo = static_cast<__nv_bfloat16*>(g.out1);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c0 + j < w.nv) {
                const size_t o = (out_row0 + (size_t)(c0 + j)) * (size_t)g.ldo + row;
                const float h = fmaxf(v[j], 0.f);
                const __nv_bfloat16 bh = __float2bfloat16_rn(h);
                hi[o] = bh;
                lo[o] = __float2bfloat16_rn(h - __bfloat162float(bh));
              }
            }
          } else {
            float* out = static_cast<float*>(g.out0) + (size_t)w.ks * g.split_stride;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c0 + j < w.nv) out[(out_row0 + (size_t)(c0 + j)) * (size_t)g.ldo + row] = v[j];
            }
          }
        }
      }
      if (from_tmem) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int gemm_tc_max_stages(int BN, int num_b) {
  const size_t stage = kABytes + (size_t)num_b * (size_t)BN * 128u;
  const size_t avail = kSmemLimit - 1024 - kBarrierArea;
  int st = (int)(avail / stage);
  return st > 12 ? 12 : st;
}

size_t gemm_tc_smem_bytes(int BN, int num_b, int stages) {
  return (size_t)stages * (kABytes + (size_t)num_b * (size_t)BN * 128u) + 1024 + kBarrierArea;
}

cudaError_t launch_gemm_tc(const GemmArgs& g, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                           const CUtensorMap& tmB1, cudaStream_t s, bool pdl) {
  auto kern = g.epi == 0   ? gemm_tc_kernel<0>
              : g.epi == 1 ? gemm_tc_kernel<1>
              : g.y_acc == 2 ? gemm_tc_kernel<3>   // combine with atomic adds
                             : gemm_tc_kernel<2>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem_bytes);
  if (err != cudaSuccess) return err;
  return launch_k(kern, dim3(g.grid), dim3(kThreads), g.smem_bytes, s, pdl, tmA, tmB0, tmB1, g);
}

}  // namespace smoe
