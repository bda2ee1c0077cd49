// The routed experts' whole FFN in one persistent launch on the tcgen05
// tensor cores: GEMM 1 (+ ReLU) and GEMM 2 (+ combine) tiles interleaved by
// blocks of experts, so each expert's hidden activations H are read back by
// GEMM 2 while they are still in L2 instead of making a round trip through
// HBM between two launches.
//
// The FFN is the two-layer bias-free MLP of each expert ("Top-1 路由 (Top-1
// Routing)", compassingai.com, key-parameter section) over the fixed-shape
// per-expert buffer ("MoE 专家容量因子与 Token 丢弃", wiblog.cn, section on
// where capacity comes from); GEMM 2's epilogue is the combine step (the
// gate scales the expert output when gate_multiply is set: the Switch
// Transformer walk-through's Switch layer, Eq. 2, against Top-1 Routing's
// step 3).  With top-2 or expert-choice routing several slots of one token
// add into its y row with atomic adds (the row starts at zero or at the
// shared expert's output).  Tile shapes, operand layouts, the hi + lo split of H and the
// epilogues are those of gemm_tc.cu (swap AB: expert weights are the
// 128-row MMA M, the expert's tokens the MMA N).
//
// Schedule.  Work items (expert, token tile) are cut into blocks of `eb`
// items; the unit list is S1(0), S1(1), S2(0), S1(2), S2(1), ..., S2(B-1),
// where S1(b) holds block b's GEMM 1 tiles (m1 per item) and S2(b) its GEMM
// 2 tiles (m2 per item).  CTAs claim units in list order from a global
// counter (GEMM 2 tiles cost about four GEMM 1 tiles, so a static split
// would be uneven); the producer lane claims and passes each claim to the
// MMA lane and the epilogue warps through a shared-memory queue.  A GEMM 2 unit needs
// every GEMM 1 tile of its item: each epilogue warp that stores a slice of
// H adds one to the item's counter, and the producer of a GEMM 2 unit
// waits (bounded) for 4 * m1 before it loads H.  Every dependency sits
// earlier in the list, was claimed earlier, and had all its copies issued
// before its CTA claimed anything else; MMAs and epilogues wait on nothing
// outside their CTA, so the earliest waiting unit's inputs always complete:
// no wait is circular.
//
// Tail split as in gemm_tc.cu, applied to the list's last GEMM 2 tiles.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace smoe {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kABytes = kTileM * 128;   // 16 KB per stage
constexpr size_t kSmemLimit = 232448;
constexpr size_t kBarrierArea = 512;
constexpr int kMaxPieces = 4;
constexpr int kMinPieceKBlocks = 4;
constexpr int kMaxAcc = 4;
constexpr int kMaxSegs = 2 * kFfnMaxBlocks;
constexpr int kQ = 16;   // claimed units in flight between the producer and the consumers

// Segment table of the schedule (shared memory, built once per CTA).
struct Segs {
  int n;
  int start[kMaxSegs + 1];
  int kind[kMaxSegs];    // 1: GEMM 1 tiles, 2: GEMM 2 tiles
  int block[kMaxSegs];
};

struct Unit {
  int kind;            // 1 or 2
  int j;               // work item (index into entries)
  int e, nt, mt, nv;   // expert, token tile, 128-row weight tile, filled columns
  int kb0, nkb;        // K blocks [kb0, kb0 + nkb)
  int unit;            // index among split pieces, -1: whole tile
  int sidx, pieces;
};

// Walks the segment table forward from *cur (positions only grow per role).
__device__ __forceinline__ void decode_unit(const FfnArgs& a, const Segs& sg, int& cur, int p,
                                            int full, int pieces, Unit& u) {
  int tile = p, piece = 0;
  u.unit = -1;
  u.sidx = 0;
  u.pieces = pieces;
  if (p >= full) {
    u.unit = p - full;
    u.sidx = u.unit / pieces;
    piece = u.unit - u.sidx * pieces;
    tile = full + u.sidx;
  }
  while (cur + 1 < sg.n && sg.start[cur + 1] <= tile) ++cur;
  const int l = tile - sg.start[cur];
  u.kind = sg.kind[cur];
  const int m = u.kind == 1 ? a.m1 : a.m2;
  u.j = sg.block[cur] * a.eb + l / m;
  u.mt = l - (l / m) * m;
  const int2 en = a.entries[u.j];
  u.e = en.x;
  u.nt = en.y;
  const int kept = min(a.counts[u.e], a.cap);
  u.nv = min(a.BN, kept - u.nt * a.BN);
  const int kbt = u.kind == 1 ? a.kb1 : a.kb2;
  if (u.unit < 0) {
    u.kb0 = 0;
    u.nkb = kbt;
  } else {
    u.kb0 = piece * kbt / pieces;
    u.nkb = (piece + 1) * kbt / pieces - u.kb0;
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
  unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 0; it < kWaitMaxIters; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 31u) == 31u && globaltimer_ns() - t0 > kWaitTimeoutNs) break;
  }
  atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *cnt reaches `target` (GEMM 1 of a work item done).
__device__ bool wait_count(const int32_t* cnt, int target, volatile int* abort_flag,
                           int* status) {
  if (ld_acquire(cnt) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (unsigned it = 1; it < kWaitMaxIters; ++it) {
    __nanosleep(64);
    if (ld_acquire(cnt) >= target) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) break;
    }
  }
  *abort_flag = 1;
  atomicExch(status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
  return false;
}

// kAtomicY: several slots add into one token's y row (top-2, expert
// choice): atomic adds, gates per slot (a separate instantiation: the
// combine loop's code size costs time).
template <bool kAtomicY>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX,
                  const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH0,
                  const __grid_constant__ CUtensorMap tmH1, const FfnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Segs sg;
  __shared__ volatile int uq[kQ];              // claimed unit positions
  __shared__ __align__(8) uint64_t q_full[kQ];   // a claim is in uq
  __shared__ __align__(8) uint64_t q_empty[kQ];  // the MMA lane and 4 epilogue warps read it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t b_bytes = (uint32_t)a.BN * 128u;
  const uint32_t stage_bytes = kABytes + 2u * b_bytes;   // sized for GEMM 2 (H hi + lo)
  const uint32_t tx1 = kABytes + b_bytes, tx2 = kABytes + 2u * b_bytes;
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)a.stages * stage_bytes);
  uint64_t* empty = full + a.stages;
  uint64_t* tfull = empty + a.stages;
  uint64_t* tempty = tfull + kMaxAcc;
  uint64_t* drain = tempty + kMaxAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t n_acc = kMaxAcc;   // BN <= 128: four 128-column accumulators
  const uint32_t tmem_cols = 512u;
  int* status = a.status;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 5);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tmW1);
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW2);
    prefetch_tensormap(&tmH0);
    prefetch_tensormap(&tmH1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) {
    // While the previous kernel finishes: pull into L2 the W1 tile this CTA
    // most likely claims first (unit blockIdx.x, taking work item j to be
    // expert j, as when every expert has one token tile).  Only a hint: a
    // wrong guess costs bandwidth, never a result.
    const int j = blockIdx.x / a.m1, mt = blockIdx.x - (blockIdx.x / a.m1) * a.m1;
    const size_t row = (size_t)j * a.F + (size_t)mt * kTileM;
    if (row + kTileM <= (size_t)a.n_experts * a.F) {
      const char* base = static_cast<const char*>(a.W1) + row * (size_t)a.d * 2;
      const uint32_t bytes = kTileM * (uint32_t)a.d * 2u;
      for (uint32_t off = 0; off < bytes; off += 32768u)
        l2_prefetch_bulk(base + off, min(32768u, bytes - off));
    }
  }
  grid_dep_wait();   // the work list, its counters and the expert buffer
  grid_dep_launch();
  if (threadIdx.x == 0) {
    // the schedule over the work list of the previous kernel
    const int ne = *a.n_entries;
    const int B = (ne + a.eb - 1) / a.eb;
    int n = 0, pos = 0;
    auto add = [&](int kind, int b) {
      const int items = min(a.eb, ne - b * a.eb);
      sg.start[n] = pos;
      sg.kind[n] = kind;
      sg.block[n] = b;
      pos += items * (kind == 1 ? a.m1 : a.m2);
      ++n;
    };
    if (B > 0) add(1, 0);
    for (int b = 1; b < B; ++b) {
      add(1, b);
      add(2, b - 1);
    }
    if (B > 0) add(2, B - 1);
    sg.start[n] = pos;
    sg.n = n;
  }
  __syncthreads();

  const int total = sg.n > 0 ? sg.start[sg.n] : 0;
  // tail split: only the list's last GEMM 2 tiles are cut
  int full_tiles = total, pieces = 1;
  {
    const int grid = (int)gridDim.x;
    const int rem = total % grid;
    const int last_seg = sg.n > 0 ? sg.start[sg.n] - sg.start[sg.n - 1] : 0;
    if (a.part && rem > 0 && 2 * rem <= grid && rem <= last_seg) {
      int p = min(min(grid / rem, a.kb2 / kMinPieceKBlocks), kMaxPieces);
      if (p >= 2 && rem * p <= a.part_units) {
        full_tiles = total - rem;
        pieces = p;
      }
    }
  }
  const int n_units = full_tiles + (total - full_tiles) * pieces;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_a = l2_policy_evict_first();   // weights: streamed once
      const uint64_t pol_b = l2_policy_evict_last();    // tokens / H: reused by every weight tile
      int cur = 0;
      uint32_t qi = 0;
      // Claims the next unit of the list (dynamic: units differ in cost) and
      // hands it to the MMA lane and the epilogue warps through uq.
      auto claim = [&](int& p) -> bool {
        const int slot = (int)(qi % kQ);
        if (!mbar_wait(&q_empty[slot], ((qi / kQ) & 1u) ^ 1u, abort_flag, status,
                       SWITCH_MOE_ERR_DEVICE_TIMEOUT))
          return false;
        p = min(atomicAdd(a.sched, 1), n_units);
        uq[slot] = p;
        mbar_arrive(&q_full[slot]);
        ++qi;
        return true;
      };
      int p = n_units;
      bool ok = claim(p);
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      while (ok && p < n_units) {
        Unit u;
        decode_unit(a, sg, cur, p, full_tiles, pieces, u);
        const bool g1 = u.kind == 1;
        const CUtensorMap* mA = g1 ? &tmW1 : &tmW2;
        const int ya = u.e * (g1 ? a.F : a.d) + u.mt * kTileM;
        const int yb = u.e * a.C + u.nt * a.BN;
        if (!g1) {
          // H of this item comes from GEMM 1 tiles on other CTAs: wait for
          // all of them before the unit's first copy is issued
          if (!wait_count(a.dep + u.j, 4 * a.m1, abort_flag, status)) break;
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int kb = 0; kb < u.nkb; ++kb) {
          uint8_t* st = tiles + (size_t)stage * stage_bytes;
          const int kx = (u.kb0 + kb) * kTileK;
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status,
                         SWITCH_MOE_ERR_DEVICE_TIMEOUT)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], g1 ? tx1 : tx2);
          tma_load_2d(st, mA, &full[stage], kx, ya, pol_a);
          if (g1) {
            tma_load_2d(st + kABytes, &tmX, &full[stage], kx, yb, pol_b);
          } else {
            tma_load_2d(st + kABytes, &tmH0, &full[stage], kx, yb, pol_b);
            tma_load_2d(st + kABytes + b_bytes, &tmH1, &full[stage], kx, yb, pol_b);
          }
          ++issued;
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ok = claim(p);
      }
      const uint32_t S = (uint32_t)a.stages;
      for (uint32_t s = 0; s < S && s < issued; ++s) {
        const uint32_t last = s + S * ((issued - 1u - s) / S);
        drain_wait(&full[s], (last / S) & 1u, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      int cur = 0;
      int stage = 0;
      uint32_t phase = 0, it = 0, qi = 0;
      bool ok = true;
      for (;; ++it) {
        const int slot = (int)(qi % kQ);
        if (!mbar_wait(&q_full[slot], (qi / kQ) & 1u, abort_flag, status,
                       SWITCH_MOE_ERR_DEVICE_TIMEOUT))
          break;
        const int p = uq[slot];
        mbar_arrive(&q_empty[slot]);
        ++qi;
        if (p >= n_units) break;
        Unit u;
        decode_unit(a, sg, cur, p, full_tiles, pieces, u);
        const uint32_t acc = it % n_acc, acc_par = (it / n_acc) & 1u;
        if (!mbar_wait(&tempty[acc], acc_par ^ 1u, abort_flag, status,
                       SWITCH_MOE_ERR_DEVICE_TIMEOUT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 128u;
        const uint32_t idesc = idesc_bf16_f32(128u, ((uint32_t)u.nv + 15u) & ~15u);
        const bool two_b = u.kind == 2;
        for (int kb = 0; kb < u.nkb; ++kb) {
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
          for (int k = 0; k < kTileK / 16; ++k) {
            const uint64_t ad = smem_desc_sw128(a_addr + (uint32_t)k * 32u);
            mma_bf16_ss(d_tmem, ad, smem_desc_sw128(b0_addr + (uint32_t)k * 32u), idesc,
                        (kb | k) != 0 ? 1u : 0u);
            if (two_b)
              mma_bf16_ss(d_tmem, ad, smem_desc_sw128(b1_addr + (uint32_t)k * 32u), idesc, 1u);
          }
          mma_commit(&empty[stage]);
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      mma_commit(drain);
      drain_wait(drain, 0u, status);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const unsigned kAll = 0xffffffffu;
    int cur = 0;
    uint32_t it = 0, qi = 0;
    for (;;) {
      const int slot = (int)(qi % kQ);
      int p = n_units;
      bool got = true;
      if (lane == 0) {
        got = mbar_wait(&q_full[slot], (qi / kQ) & 1u, abort_flag, status,
                        SWITCH_MOE_ERR_DEVICE_TIMEOUT);
        if (got) {
          p = uq[slot];
          mbar_arrive(&q_empty[slot]);
        }
      }
      ++qi;
      got = __shfl_sync(kAll, got, 0);
      p = __shfl_sync(kAll, p, 0);
      if (!got || p >= n_units) break;
      Unit u;
      decode_unit(a, sg, cur, p, full_tiles, pieces, u);
      const uint32_t my_it = it++;
      const uint32_t acc = my_it % n_acc, acc_par = (my_it / n_acc) & 1u;
      const bool g1 = u.kind == 1;
      const int row = u.mt * kTileM + q * 32 + lane;   // weight row = output column
      const bool row_ok = row < (g1 ? a.F : a.d);
      const size_t out_row0 = (size_t)u.e * a.C + (size_t)u.nt * a.BN;
      auto tok_gate = [&](int c, int& tk, float& gv) {
        tk = 0;
        gv = 1.f;
        if (c + lane < u.nv) {
          tk = a.tok_of_slot[out_row0 + (size_t)(c + lane)];
          if (a.gate_multiply)   // several slots per token: the gate belongs to the slot
            gv = kAtomicY ? a.slot_gate[out_row0 + (size_t)(c + lane)] : a.gate[tk];
        }
      };
      int tk32 = 0;
      float gv32 = 1.f;
      if (!g1 && u.unit < 0) tok_gate(0, tk32, gv32);   // overlaps the wait below
      const bool ready =
          mbar_wait(&tfull[acc], acc_par, abort_flag, status, SWITCH_MOE_ERR_DEVICE_TIMEOUT);
      if (!__all_sync(kAll, ready)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 128u;

      const size_t tile_elems = (size_t)kTileM * (size_t)a.BN;
      bool from_tmem = true;
      const float* p0 = nullptr;
      if (u.unit >= 0) {
        // one K piece of a split GEMM 2 tile: park the partial, [column][128 rows]
        float* mine = a.part + (size_t)u.unit * tile_elems + q * 32 + lane;
        for (int c0 = 0; c0 < u.nv; c0 += 16) {
          float v[16];
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (c0 + jj < u.nv) mine[(size_t)(c0 + jj) * kTileM] = v[jj];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          int32_t* cnt = a.split_cnt + u.sidx * 4 + q;
          last = atomicAdd(cnt, 1) == u.pieces - 1;
          if (last) *cnt = 0;
        }
        if (!__shfl_sync(kAll, last, 0)) continue;
        __threadfence();
        from_tmem = false;
        p0 = a.part + (size_t)u.sidx * u.pieces * tile_elems + q * 32 + lane;
        tok_gate(0, tk32, gv32);
      }
      auto fetch16 = [&](int c0, float (&v)[16]) {
        if (from_tmem) {
          tmem_ld_32x32b_x16(taddr + (uint32_t)c0, v);
          return;
        }
        float t[kMaxPieces][16];
#pragma unroll
        for (int i = 0; i < kMaxPieces; ++i) {
          const float* src = p0 + (size_t)i * tile_elems + (size_t)c0 * kTileM;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            t[i][jj] = (i < u.pieces && c0 + jj < u.nv) ? __ldcg(src + jj * kTileM) : 0.f;
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] = t[0][jj];
#pragma unroll
        for (int i = 1; i < kMaxPieces; ++i) {
          if (i < u.pieces) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) v[jj] = v[jj] + t[i][jj];
          }
        }
      };

      if (g1) {
        // relu, then H as an unevaluated bf16 pair hi + lo
        for (int c0 = 0; c0 < u.nv; c0 += 16) {
          float v[16];
          fetch16(c0, v);
          if (!row_ok) continue;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (c0 + jj < u.nv) {
              const size_t o = (out_row0 + (size_t)(c0 + jj)) * (size_t)a.F + row;
              const float h = fmaxf(v[jj], 0.f);
              const __nv_bfloat16 bh = __float2bfloat16_rn(h);
              a.H0[o] = bh;
              a.H1[o] = __float2bfloat16_rn(h - __bfloat162float(bh));
            }
          }
        }
        // this warp's slice of the item's H is stored: publish it
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) atomicAdd(a.dep + u.j, 1);
      } else {
        // combine: y[token] = g_token * D (+ y[token]), 32 columns per step
        for (int c0 = 0; c0 < u.nv; c0 += 32) {
          if (c0 > 0) tok_gate(c0, tk32, gv32);
          float v[2][16];
          fetch16(c0, v[0]);
          fetch16(c0 + 16, v[1]);
          if constexpr (kAtomicY) {
            add_block_v4(v, tk32, gv32, a.y, a.d, u.mt * kTileM + q * 32, a.d, c0, u.nv, lane);
            continue;
          }
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int tj = __shfl_sync(kAll, tk32, jj);
            const float gj = __shfl_sync(kAll, gv32, jj);
            if (row_ok && c0 + jj < u.nv) {
              float* dst = a.y + (size_t)tj * (size_t)a.d + row;
              const float val = gj * v[jj >> 4][jj & 15];
              if constexpr (kAtomicY) {
                atomicAdd(dst, val);   // several slots add into one row
              } else {
                *dst = a.y_acc ? *dst + val : val;
              }
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

int ffn_tc_stages(int BN) {
  const size_t stage = kABytes + 2u * (size_t)BN * 128u;
  // static shared memory: the schedule table and the claim queue
  const size_t avail = kSmemLimit - 1024 - kBarrierArea - sizeof(Segs) - 1024;
  int st = (int)(avail / stage);
  return st > 12 ? 12 : st;
}

size_t ffn_tc_smem_bytes(int BN, int stages) {
  return (size_t)stages * (kABytes + 2u * (size_t)BN * 128u) + 1024 + kBarrierArea;
}

cudaError_t launch_ffn_tc(const FfnArgs& a, const CUtensorMap& tmW1, const CUtensorMap& tmX,
                          const CUtensorMap& tmW2, const CUtensorMap& tmH0,
                          const CUtensorMap& tmH1, cudaStream_t s, bool pdl) {
  auto kern = a.y_acc == 2 ? ffn_tc_kernel<true> : ffn_tc_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)a.smem_bytes);
  if (err != cudaSuccess) return err;
  return launch_k(kern, dim3(a.grid), dim3(kThreads), a.smem_bytes, s, pdl, tmW1, tmX, tmW2,
                  tmH0, tmH1, a);
}

}  // namespace smoe
