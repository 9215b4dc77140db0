// Blockwise exact attention with online softmax on the sm_103a tensor cores.
//
// One thread block owns 256 query rows (two 128-row tiles Q0, Q1) of one
// rank and one query head, and walks the key/value tiles of the ring steps
// [t_begin, t_end) in ring order: at step t it reads the shard of rank
// (rank - t) mod c ("06 - Sequence / Context Parallelism", section 4: the
// block a rank holds after t SEND/RECV rounds).  For every key tile it
//   S_h = Q_h K^T                         (tcgen05.mma, fp32 in tensor memory)
//   m'  = max(m, rowmax(scale*log2e*S_h)) (causal mask by global position)
//   P_h = 2^(scale*log2e*S_h - m')        (bf16, written back to tensor memory)
//   l   = 2^(m - m') l + rowsum(P_h)
//   O_h = 2^(m - m') O_h + P_h V          (tcgen05.mma, fp32 in tensor memory)
// which is the online-softmax update with rescaling of the earlier sums
// whenever a block raises the running maximum (quiz "Sequence Parallelism and
// Ring Attention", questions 3 and 7).  Key tiles wholly in the future of
// both query tiles are skipped; tiles that straddle the diagonal are masked
// element by element.  At the end the state is either written out (per-step
// mode) or normalised, out = O / l and lse = ln2 (m + log2 l).
//
// Warp roles (352 threads):
//   warps 0-3  softmax for Q0 (warp w reads tensor-memory lanes 32w..32w+31)
//   warps 4-7  softmax for Q1
//   warp 8     TMA loads of Q and the K tiles
//   warp 9     TMA loads of the V tiles
//   warp 10    tensor-memory allocation and the tcgen05.mma issue loop (the
//              whole warp runs it; one elected lane issues each instruction)
// Pipelines: K and V each have 2 shared-memory stages; the two query tiles
// ping-pong so that the tensor core multiplies one tile while the softmax of
// the other runs.  Tensor memory (512 columns): S0 | S1 | O0 | O1, with P_h
// stored as packed bf16 over the first 64 columns of S_h.
//
// Every mbarrier wait is bounded (ra_wait.cuh, 4 s); a wait that runs out raises an abort
// flag in shared memory and a bit in the device error word, every role
// leaves its loop, outstanding tensor-core work and TMA loads are drained
// (bounded), tensor memory is freed and the block exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>

#include "ra_internal.h"
#include "ra_wait.cuh"
#include "sm103_ptx.cuh"

namespace ra {
namespace {

constexpr int kWarpK = 8;
constexpr int kWarpV = 9;
constexpr int kWarpMma = 10;
constexpr int kThreads = 11 * 32;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Smem {
  static constexpr int kTileBytes = kTile * D * 2;   // one 128-row bf16 tile
  static constexpr int kBox = 64;                    // columns per TMA box (128 bytes)
  static constexpr int kBoxBytes = kTile * kBox * 2;
  static constexpr int kBoxes = D / kBox;
  static constexpr int KST = 2;
  static constexpr int VST = 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + KST * kTileBytes;
  static constexpr int kBar = kV + VST * kTileBytes;
  static constexpr int bQ = 0;
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + KST;
  static constexpr int bVFull = bKEmpty + KST;
  static constexpr int bVEmpty = bVFull + VST;
  static constexpr int bSFull = bVEmpty + VST;
  static constexpr int bPFull = bSFull + 2;
  static constexpr int bOFinal = bPFull + 2;
  static constexpr int bDrain = bOFinal + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kRange = kMisc + 16;          // (min, max) key position per key tile
  static constexpr int kMaxRanges = 2048;
  static constexpr int kBytes = kRange + kMaxRanges * 8;
  static constexpr int kDynamic = kBytes + 1024;     // room to align the base to 1024
  static_assert(kDynamic <= 232448, "shared memory budget");
};

// Tensor-memory column of each accumulator.
__device__ __forceinline__ uint32_t col_S(int h) { return static_cast<uint32_t>(h * 128); }
__device__ __forceinline__ uint32_t col_O(int h) { return static_cast<uint32_t>(256 + h * 128); }

// Warp-cooperative min and max of count >= 0 positions (INT_MAX / INT_MIN if empty).
__device__ __forceinline__ void warp_minmax(const int32_t* pos, int count, int lane, int& mn,
                                            int& mx) {
  mn = INT_MAX;
  mx = INT_MIN;
  for (int i = lane; i < count; i += 32) {
    const int p = __ldg(pos + i);
    mn = min(mn, p);
    mx = max(mx, p);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
}

// What a block needs to know about its two query tiles.
struct QTiles {
  int valid[2];   // rows of each tile inside the rank's shard
  int mn[2], mx[2];
  int mx_all;     // max position over both tiles
};

__device__ __forceinline__ QTiles q_tiles(const AttnParams& p, int rank, int row0, int lane) {
  QTiles q;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int start = row0 + hh * kTile;
    q.valid[hh] = max(0, min(kTile, p.n_q - start));
    warp_minmax(p.q_pos + static_cast<long long>(rank) * p.n_q + start, q.valid[hh], lane,
                q.mn[hh], q.mx[hh]);
  }
  q.mx_all = max(q.mx[0], q.mx[1]);
  return q;
}

struct KTile {
  int valid, mn, mx;
  bool skip;   // hidden from both query tiles
};

// Key tile kt of shard `src`.  `rs` holds the (min, max) positions of the
// tiles of this step in shared memory, or is null (then they are reduced
// from the positions by the calling warp).
__device__ __forceinline__ KTile k_tile(const AttnParams& p, int src, int kt, const QTiles& q,
                                        int lane, const int2* rs) {
  KTile k;
  const int start = kt * kTile;
  k.valid = min(kTile, p.n_k - start);
  if (rs != nullptr) {
    const int2 r = rs[kt];
    k.mn = r.x;
    k.mx = r.y;
  } else {
    warp_minmax(p.k_pos + static_cast<long long>(src) * p.n_k + start, k.valid, lane, k.mn, k.mx);
  }
  k.skip = p.causal ? (k.mn > q.mx_all) : (q.valid[0] + q.valid[1] == 0);
  return k;
}

// Key tile kt of shard `src` as seen by a single thread: the staged ranges,
// else the ranges in global memory, else a serial reduction of the positions.
__device__ __forceinline__ KTile k_tile_1(const AttnParams& p, int src, int kt, const QTiles& q,
                                          int ktiles, const int2* rs) {
  KTile k;
  const int start = kt * kTile;
  k.valid = min(kTile, p.n_k - start);
  if (rs != nullptr) {
    const int2 r = rs[kt];
    k.mn = r.x;
    k.mx = r.y;
  } else if (p.k_ranges != nullptr) {
    const int2 r = p.k_ranges[static_cast<long long>(src) * ktiles + kt];
    k.mn = r.x;
    k.mx = r.y;
  } else {
    const int32_t* pos = p.k_pos + static_cast<long long>(src) * p.n_k + start;
    k.mn = INT_MAX;
    k.mx = INT_MIN;
    for (int i = 0; i < k.valid; ++i) {
      const int v = __ldg(pos + i);
      k.mn = min(k.mn, v);
      k.mx = max(k.mx, v);
    }
  }
  k.skip = p.causal ? (k.mn > q.mx_all) : (q.valid[0] + q.valid[1] == 0);
  return k;
}

__device__ __forceinline__ int ring_src(int rank, int t, int c) {
  int s = (rank - t) % c;
  return s < 0 ? s + c : s;
}

// Key/value shard read at step t: the ring's (rank - t) mod c, or, in the
// all-gather form, the whole gathered buffer (source 0, c*n_k rows).
__device__ __forceinline__ int step_src(const AttnParams& p, int rank, int t) {
  return p.kv_all ? 0 : ring_src(rank, t, p.c);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  // Align the shared-window address (not the generic one) to 1024 bytes, as
  // the 128-byte swizzle pattern repeats every 1024 bytes.
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const Abort ab{abort_flag, p.err};

  // taken from lane 0 so that the compiler can keep it in a uniform register
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;

  // ---- which problem this block owns -----------------------------------
  // Blocks start roughly in the order of their linear index: (batch, key/value
  // head) outermost, then the query blocks (heaviest first), then the G query
  // heads sharing the key/value head, so that the blocks in flight together
  // read the keys and values of one head, which stay in L2.
  const long long lin = static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x;
  const int hl = static_cast<int>(lin % p.G);
  const long long rest = lin / p.G;
  int yb = static_cast<int>(rest % gridDim.y);
  const int bg = static_cast<int>(rest / gridDim.y);
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int h = g * p.G + hl;
  if (p.block_order != nullptr) yb = p.block_order[yb];
  const int rank = yb / p.q_blocks_per_rank;
  const int row0 = (yb % p.q_blocks_per_rank) * kPairRows;   // local row of Q0
  const int ktiles = (p.n_k + kTile - 1) / kTile;

  // ---- set-up ----------------------------------------------------------
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bQ), 1);
    for (int s = 0; s < L::KST; ++s) {
      ptx::mbar_init(bar(L::bKFull + s), 1);
      ptx::mbar_init(bar(L::bKEmpty + s), 1);
    }
    for (int s = 0; s < L::VST; ++s) {
      ptx::mbar_init(bar(L::bVFull + s), 1);
      ptx::mbar_init(bar(L::bVEmpty + s), 1);
    }
    for (int hh = 0; hh < 2; ++hh) {
      ptx::mbar_init(bar(L::bSFull + hh), 1);
      ptx::mbar_init(bar(L::bPFull + hh), 128);
    }
    ptx::mbar_init(bar(L::bOFinal), 1);
    ptx::mbar_init(bar(L::bDrain), 1);
    // A device error left by an earlier block or launch: do no work.
    *abort_flag = (*reinterpret_cast<volatile unsigned int*>(p.err) != 0) ? 1 : 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpK && lane == 0) {
    ptx::tma_prefetch_desc(&tm_q);
    ptx::tma_prefetch_desc(&tm_k);
  }
  if (warp == kWarpV && lane == 0) ptx::tma_prefetch_desc(&tm_v);
  if (warp == kWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  // Stage the (min, max) key position of every key tile this block visits.
  int2* const ranges = reinterpret_cast<int2*>(smem + L::kRange);
  const int nsteps = p.t_end - p.t_begin;
  const bool staged = static_cast<long long>(nsteps) * ktiles <= L::kMaxRanges;
  if (staged) {
    const int total = nsteps * ktiles;
    if (p.k_ranges != nullptr) {
      for (int i = threadIdx.x; i < total; i += kThreads) {
        const int src = step_src(p, rank, p.t_begin + i / ktiles);
        ranges[i] = p.k_ranges[static_cast<long long>(src) * ktiles + i % ktiles];
      }
    } else {
      for (int i = warp; i < total; i += kThreads / 32) {
        const int src = step_src(p, rank, p.t_begin + i / ktiles);
        const int kt = i % ktiles;
        int mn, mx;
        warp_minmax(p.k_pos + static_cast<long long>(src) * p.n_k + kt * kTile,
                    min(kTile, p.n_k - kt * kTile), lane, mn, mx);
        if (lane == 0) ranges[i] = make_int2(mn, mx);
      }
    }
  }
  auto step_ranges = [&](int t) -> const int2* {
    return staged ? ranges + (t - p.t_begin) * ktiles : nullptr;
  };
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const QTiles qt = q_tiles(p, rank, row0, lane);

  if (warp == kWarpK || warp == kWarpV) {
    // ===================== TMA producers ================================
    const bool is_k = (warp == kWarpK);
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const int nst = is_k ? L::KST : L::VST;
    const int full0 = is_k ? L::bKFull : L::bVFull;
    const int empty0 = is_k ? L::bKEmpty : L::bVEmpty;
    const uint32_t stage0 = sbase + (is_k ? L::kK : L::kV);
    const bool q_issued = is_k && !*abort_flag;
    if (q_issued && lane == 0) {
      // Q tiles are read by this block only: their lines go first when L2
      // needs room, which keeps the key and value tiles (read by every
      // block) resident
      const uint64_t pol = ptx::l2_policy_evict_first();
      ptx::mbar_arrive_expect_tx(bar(L::bQ), 2 * L::kTileBytes);
      for (int hh = 0; hh < 2; ++hh)
        for (int x = 0; x < L::kBoxes; ++x)
          ptx::tma_load_4d_hint(sbase + L::kQ + hh * L::kTileBytes + x * L::kBoxBytes, &tm_q,
                                bar(L::bQ), x * L::kBox, h, rank * p.n_q + row0 + hh * kTile, b, pol);
    }
    uint32_t j = 0;
    bool ok = !*abort_flag;
    for (int t = p.t_begin; t < p.t_end && ok; ++t) {
      const int src = step_src(p, rank, t);
      const int2* rs = step_ranges(t);
      for (int kt = 0; kt < ktiles; ++kt) {
        const KTile k = k_tile(p, src, kt, qt, lane, rs);
        if (k.skip) continue;
        if (lane == 0) {
          const int s = static_cast<int>(j % nst);
          const uint32_t n = j / nst;
          if (n > 0) ok = wait_bar(bar(empty0 + s), (n - 1) & 1u, ab, kErrTimeoutEmpty);
          if (ok) {
            ptx::mbar_arrive_expect_tx(bar(full0 + s), L::kTileBytes);
            for (int x = 0; x < L::kBoxes; ++x)
              ptx::tma_load_4d(stage0 + s * L::kTileBytes + x * L::kBoxBytes, map,
                               bar(full0 + s), x * L::kBox, g,
                               (p.kv_by_holder ? rank : src) * p.n_k + kt * kTile, b);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++j;
      }
    }
    if (lane == 0 && *abort_flag) {
      // Let the loads still in flight land before the block exits.
      if (q_issued) wait_bar_drain(bar(L::bQ), 0);
      for (int s = 0; s < nst; ++s) {
        const uint32_t issued = (j > static_cast<uint32_t>(s)) ? (j - 1 - s) / nst + 1 : 0;
        if (issued > 0) wait_bar_drain(bar(full0 + s), (issued - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ===================== tensor-core issue ============================
    // The whole warp runs this loop with the same values in every lane, so
    // the descriptors and addresses stay warp-uniform; one elected lane
    // issues each tcgen05.mma / commit (no branch around the issue), and the
    // waits are made warp-uniform.  tcgen05.mma issue holds the issuing lane
    // until the tensor core takes the instruction, so everything between two
    // batches is kept short.
    {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(128, 128, false);
      constexpr uint32_t idPV = ptx::idesc_bf16_f32(128, D, true);
      bool ok = __all_sync(0xffffffffu, wait_bar(bar(L::bQ), 0, ab, kErrTimeoutQ));
      bool issued_any = false;
      // Shared-memory descriptors of the first Q tile / K stage / V stage;
      // the others differ only in the 16-byte address field (bits 0-13).
      const uint64_t dQ = ptx::smem_desc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dK = ptx::smem_desc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dV = ptx::smem_desc_sw128(sbase + L::kV, L::kBoxBytes, 1024);
      auto issue_S = [&](int hh, int ks) {
        const uint64_t qd = dQ + static_cast<uint64_t>((hh * L::kTileBytes) >> 4);
        const uint64_t kd = dK + static_cast<uint64_t>((ks * L::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk / 4) * L::kBoxBytes + (kk % 4) * 32) >> 4);
          ptx::tc_mma_ss_elect(tmem + col_S(hh), qd + o, kd + o, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_PV = [&](int hh, int vs) {
        const uint64_t vd = dV + static_cast<uint64_t>((vs * L::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          ptx::tc_mma_ts_elect(tmem + col_O(hh), tmem + col_S(hh) + kk * 8,
                         vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), idPV, 1u);
      };

      uint32_t j = 0;
      for (int t = p.t_begin; t < p.t_end && ok; ++t) {
        const int src = step_src(p, rank, t);
        const int2* rs = step_ranges(t);
        unsigned long long nfull = 0, npart = 0, nskip = 0;
        for (int kt = 0; kt < ktiles; ++kt) {
          const KTile k = k_tile_1(p, src, kt, qt, ktiles, rs);
          if (p.work != nullptr) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              if (qt.valid[hh] == 0) continue;
              if (!p.causal || k.mx <= qt.mn[hh]) ++nfull;
              else if (k.mn > qt.mx[hh]) ++nskip;
              else ++npart;
            }
          }
          if (k.skip) continue;
          const int ks = static_cast<int>(j % L::KST);
          ok = __all_sync(0xffffffffu, wait_bar(bar(L::bKFull + ks), (j / L::KST) & 1u, ab, kErrTimeoutK));
          if (!ok) break;
          ptx::tc_fence_after_sync();
          if (j == 0) {
            for (int hh = 0; hh < 2; ++hh) {
              issue_S(hh, ks);
              ptx::tc_commit_elect(bar(L::bSFull + hh));
            }
            issued_any = true;
          } else {
            const uint32_t jp = j - 1;
            const int vs = static_cast<int>(jp % L::VST);
            ok = __all_sync(0xffffffffu, wait_bar(bar(L::bVFull + vs), (jp / L::VST) & 1u, ab, kErrTimeoutV));
            for (int hh = 0; hh < 2 && ok; ++hh) {
              ok = __all_sync(0xffffffffu, wait_bar(bar(L::bPFull + hh), jp & 1u, ab, kErrTimeoutP));
              if (!ok) break;
              ptx::tc_fence_after_sync();
              issue_PV(hh, vs);
              issue_S(hh, ks);
              ptx::tc_commit_elect(bar(L::bSFull + hh));
            }
            if (ok) ptx::tc_commit_elect(bar(L::bVEmpty + vs));
          }
          if (!ok) break;
          ptx::tc_commit_elect(bar(L::bKEmpty + ks));
          ++j;
        }
        if (p.work != nullptr && ok && lane == 0) {
          ra_work* w = p.work + static_cast<long long>(rank) * p.c + t;
          atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_full), nfull);
          atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_partial), npart);
          atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_skipped), nskip);
        }
      }
      if (ok && j > 0) {
        const uint32_t jp = j - 1;
        const int vs = static_cast<int>(jp % L::VST);
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::bVFull + vs), (jp / L::VST) & 1u, ab, kErrTimeoutV));
        for (int hh = 0; hh < 2 && ok; ++hh) {
          ok = __all_sync(0xffffffffu, wait_bar(bar(L::bPFull + hh), jp & 1u, ab, kErrTimeoutP));
          if (!ok) break;
          ptx::tc_fence_after_sync();
          issue_PV(hh, vs);
        }
        if (ok) ptx::tc_commit_elect(bar(L::bOFinal));
      }
      if (!ok && issued_any) {
        // Drain the tensor core before tensor memory is released.
        ptx::tc_commit_elect(bar(L::bDrain));
        if (!wait_bar_drain(bar(L::bDrain), 0)) raise_error(p.err, kErrTimeoutDrain);
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax warpgroups ===========================
    const int hh = warp >> 2;                 // query tile of this warpgroup
    const int wq = warp & 3;                  // lane quarter of tensor memory
    const int r = wq * 32 + lane;             // row inside the tile
    const int local_row = row0 + hh * kTile + r;
    const bool row_ok = r < qt.valid[hh];
    const long long qrow = static_cast<long long>(rank) * p.n_q + local_row;
    const long long R = static_cast<long long>(p.c) * p.n_q;
    const int qpos = row_ok ? __ldg(p.q_pos + qrow) : INT_MIN;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + col_S(hh);
    const uint32_t tO = tmem + lane_base + col_O(hh);
    const float sl2 = p.scale_log2;

    float m_run = -INFINITY;
    float l_run = 0.f;
    {
      // Initial state: loaded (per-step mode) or empty.
      const float* src_o = nullptr;
      if (p.load_state && row_ok) {
        const long long si = (static_cast<long long>(b) * p.Hq + h) * R + qrow;
        m_run = p.m_state[si];
        l_run = p.l_state[si];
        src_o = p.o_state + ((static_cast<long long>(b) * R + qrow) * p.Hq + h) * D;
      }
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t u[32];
        if (src_o != nullptr) {
          const float4* s4 = reinterpret_cast<const float4*>(src_o + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = s4[i];
            u[4 * i + 0] = __float_as_uint(f.x);
            u[4 * i + 1] = __float_as_uint(f.y);
            u[4 * i + 2] = __float_as_uint(f.z);
            u[4 * i + 3] = __float_as_uint(f.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        ptx::tmem_st32(tO + cc * 32, u);
      }
      ptx::tmem_wait_st();
    }

    uint32_t j = 0;
    bool ok = true;
    for (int t = p.t_begin; t < p.t_end && ok; ++t) {
      const int src = step_src(p, rank, t);
      const int2* rs = step_ranges(t);
      const int32_t* kpos_src = p.k_pos + static_cast<long long>(src) * p.n_k;
      unsigned long long pairs = 0;
      for (int kt = 0; kt < ktiles; ++kt) {
        const KTile k = k_tile(p, src, kt, qt, lane, rs);
        if (k.skip) continue;
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::bSFull + hh), j & 1u, ab, kErrTimeoutS));
        if (!ok) break;
        ptx::tc_fence_after_sync();
        const bool masked = (k.valid < kTile) || (p.causal && k.mx > qt.mn[hh]);
        const int32_t* kp = kpos_src + kt * kTile;

        // visibility of each key column (partial tiles only), before S is loaded
        uint32_t bits[4] = {~0u, ~0u, ~0u, ~0u};
        unsigned int nvis = static_cast<unsigned int>(k.valid);
        if (masked && p.k_sorted) {
          // positions increase inside the tile: the visible keys are the prefix
          // of those at or before this row's position (binary search)
          int cnt = k.valid;
          if (p.causal) {
            cnt = 0;
#pragma unroll
            for (int step = 128; step > 0; step >>= 1)
              if (cnt + step <= k.valid && __ldg(kp + cnt + step - 1) <= qpos) cnt += step;
          }
          nvis = static_cast<unsigned int>(cnt);
#pragma unroll
          for (int w = 0; w < 4; ++w)
            bits[w] = cnt >= 32 * (w + 1) ? ~0u : (cnt > 32 * w ? (1u << (cnt - 32 * w)) - 1u : 0u);
        } else if (masked) {
          nvis = 0;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t bb = 0;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
              const int col = cc * 32 + i;
              const bool vis = col < k.valid && (!p.causal || __ldg(kp + min(col, k.valid - 1)) <= qpos);
              bb |= (vis ? 1u : 0u) << i;
            }
            bits[cc] = bb;
            nvis += __popc(bb);
          }
        }
        uint32_t sv[128];
        float mx;
        if (!masked) {
          // every key visible: the tensor-memory load itself forms the row
          // maximum (tcgen05.ld.red, sm_103a)
          ptx::tmem_ld128_max(tS, sv, mx);
        } else {
          ptx::tmem_ld128(tS, sv);
          // hidden or padding keys become -inf before the max and the exponent
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (!((bits[i >> 5] >> (i & 31)) & 1u)) sv[i] = 0xff800000u;
          // row maximum: eight independent chains of three-input max
          float mc[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            mc[c] = ptx::fmax3(__uint_as_float(sv[16 * c]), __uint_as_float(sv[16 * c + 1]),
                               __uint_as_float(sv[16 * c + 2]));
#pragma unroll
          for (int i = 3; i < 15; i += 2) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              mc[c] = ptx::fmax3(mc[c], __uint_as_float(sv[16 * c + i]), __uint_as_float(sv[16 * c + i + 1]));
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) mc[c] = fmaxf(mc[c], __uint_as_float(sv[16 * c + 15]));
          mx = ptx::fmax3(ptx::fmax3(mc[0], mc[1], mc[2]), ptx::fmax3(mc[3], mc[4], mc[5]),
                          fmaxf(mc[6], mc[7]));
        }
        const float m_new = fmaxf(m_run, mx * sl2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;

        // rescale the accumulator when the running maximum rose; the previous
        // P.V has completed (this tile's S was committed after it), and the
        // next one is issued only after this tile's P is handed over
        const float alpha = (m_run == m_new) ? 1.f : ptx::ex2(m_run - m_new);
        if (__any_sync(0xffffffffu, (alpha != 1.f) && (m_run != -INFINITY))) {
          const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll 1
          for (int half = 0; half < D / 64; ++half) {
            uint32_t u[64];
            ptx::tmem_ld64(tO + half * 64, u);
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
              float y0, y1;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(u[i]), __uint_as_float(u[i + 1])), a2),
                             y0, y1);
              u[i] = __float_as_uint(y0);
              u[i + 1] = __float_as_uint(y1);
            }
            uint32_t w0[32], w1[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              w0[i] = u[i];
              w1[i] = u[32 + i];
            }
            ptx::tmem_st32(tO + half * 64, w0);
            ptx::tmem_st32(tO + half * 64 + 32, w1);
          }
        }

        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
        const uint64_t negm2 = ptx::f2_pack(-m_use, -m_use);
        uint64_t acc = ptx::f2_pack(0.f, 0.f);
        uint64_t acc1 = ptx::f2_pack(0.f, 0.f);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t sh[64];
          ptx::tmem_ld64(tS + half * 64, sh);
          if (masked) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (!((bits[half * 2 + (i >> 5)] >> (i & 31)) & 1u)) sh[i] = 0xff800000u;
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t x = ptx::f2_fma(ptx::f2_pack(__uint_as_float(sh[cc * 32 + 2 * i]),
                                                          __uint_as_float(sh[cc * 32 + 2 * i + 1])),
                                             sl2x2, negm2);
              float x0, x1;
              ptx::f2_unpack(x, x0, x1);
              const float e0 = ptx::ex2(x0);
              const float e1 = ptx::ex2(x1);
              if (i & 1) acc1 = ptx::f2_add(acc1, ptx::f2_pack(e0, e1));
              else acc = ptx::f2_add(acc, ptx::f2_pack(e0, e1));
              pk[i] = ptx::pack_bf16x2(e0, e1);
            }
            ptx::tmem_st16(tS + half * 32 + cc * 16, pk);
          }
        }
        float sm0, sm1;
        ptx::f2_unpack(ptx::f2_add(acc, acc1), sm0, sm1);
        const float sum = sm0 + sm1;
        l_run = l_run * alpha + sum;
        m_run = m_new;
        if (row_ok) pairs += nvis;
        ptx::tmem_wait_st();
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(bar(L::bPFull + hh));
        ++j;
      }
      if (p.work != nullptr && ok) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
        if (lane == 0 && pairs > 0) {
          ra_work* w = p.work + static_cast<long long>(rank) * p.c + t;
          atomicAdd(reinterpret_cast<unsigned long long*>(&w->pairs), pairs);
        }
      }
    }

    // ---- epilogue ---------------------------------------------------------
    if (ok && j > 0) ok = __all_sync(0xffffffffu, wait_bar(bar(L::bOFinal), 0, ab, kErrTimeoutO));
    if (ok) {
      ptx::tc_fence_after_sync();
      if (p.finalize) {
        const int orow = row_ok ? qpos : 0;
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        const long long obase = ((static_cast<long long>(b) * p.S_out + orow) * p.Hq + h) * D;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          ptx::tmem_ld32(tO + cc * 32, u);
          if (row_ok && p.out_f32) {
            float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(u[4 * i]) * inv_l, __uint_as_float(u[4 * i + 1]) * inv_l,
                                  __uint_as_float(u[4 * i + 2]) * inv_l, __uint_as_float(u[4 * i + 3]) * inv_l);
          } else if (row_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + obase + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 0]) * inv_l, __uint_as_float(u[8 * i + 1]) * inv_l);
              w.y = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv_l, __uint_as_float(u[8 * i + 3]) * inv_l);
              w.z = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv_l, __uint_as_float(u[8 * i + 5]) * inv_l);
              w.w = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv_l, __uint_as_float(u[8 * i + 7]) * inv_l);
              d4[i] = w;
            }
          }
        }
        if (row_ok && p.lse != nullptr) {
          const float lse = (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
          p.lse[(static_cast<long long>(b) * p.Hq + h) * p.S_out + orow] = lse;
        }
      }
      if (p.store_state) {
        float* dst = p.o_state + ((static_cast<long long>(b) * R + qrow) * p.Hq + h) * D;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          ptx::tmem_ld32(tO + cc * 32, u);
          if (row_ok) {
            float4* d4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                  __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
          }
        }
        if (row_ok) {
          const long long si = (static_cast<long long>(b) * p.Hq + h) * R + qrow;
          p.m_state[si] = m_run;
          p.l_state[si] = l_run;
        }
      }
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.

template <int D>
int launch_d(const AttnParams& p, const void* q, const void* k, const void* v,
             long long q_rows_total, long long k_rows_total, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  std::memset(&mq, 0, sizeof(mq));
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  launch_stage() = "cuTensorMapEncodeTiled";
  int e = make_tma_map_bf16(&mq, q, p.B, q_rows_total, p.Hq, D, kTile);
  if (!e) e = make_tma_map_bf16(&mk, k, p.B, k_rows_total, p.Hkv, D, kTile);
  if (!e) e = make_tma_map_bf16(&mv, v, p.B, k_rows_total, p.Hkv, D, kTile);
  if (e) return e;
  const int smem = Smem<D>::kDynamic;
  launch_stage() = "cudaFuncSetAttribute (tensor-core kernel)";
  cudaError_t ce = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (ce != cudaSuccess) return static_cast<int>(ce);
  const int yb = (p.y_blocks > 0) ? p.y_blocks : p.c * p.q_blocks_per_rank;
  dim3 grid(static_cast<unsigned>(p.B * p.Hq), static_cast<unsigned>(yb));
  launch_stage() = "tensor-core kernel launch";
  attn_fwd_tc_kernel<D><<<grid, kThreads, smem, stream>>>(mq, mk, mv, p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_attn_tc(const AttnParams& p, const void* q, const void* k, const void* v,
                   long long q_rows_total, long long k_rows_total, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // D = 128 runs on SM pairs (attn_pair_sm103.cu); D = 64 on single CTAs
  if (p.D == 128) return launch_attn_pair(p, q, k, v, q_rows_total, k_rows_total, stream);
  if (p.D == 64) return launch_d<64>(p, q, k, v, q_rows_total, k_rows_total, s);
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace ra
