// Blockwise exact attention with online softmax on pairs of sm_103a SMs.
//
// The computation of the single-CTA kernel (attn_tc_sm103.cu): for every
// key tile of the ring steps [t_begin, t_end), in ring order (at step t the
// shard of rank (rank - t) mod c, "06 - Sequence / Context Parallelism",
// section 4),
//   S  = Q K^T                           (fp32, tensor memory)
//   m' = max(m, rowmax(scale*log2e*S))   (causal mask by global position)
//   P  = 2^(scale*log2e*S - m')          (bf16)
//   l  = 2^(m - m') l + rowsum(P)
//   O  = 2^(m - m') O + P V
// the online-softmax update with rescaling whenever a block raises the
// running maximum (quiz "Sequence Parallelism and Ring Attention", questions
// 3 and 7); then out = O / l and lse = ln2 (m + log2 l), or the state written
// back (per-step mode).
//
// A thread-block cluster of two CTAs shares the tensor cores of two SMs.
// The pair owns 512 query rows: two 128-row tiles in each CTA.  Every product
// is a pair instruction (tcgen05.mma.cta_group::2, M = 256: tile h of both
// CTAs) issued by the even CTA.  Each CTA stages only half of every key tile
// (64 keys: the B operand of S = Q K^T is split along N) and half of every
// value tile (64 of the 128 value columns: the B operand of O += P V).
//
// Tensor memory per CTA (512 columns): O0 | S0 | O1 | S1.  P goes to shared
// memory (the A operand of P V), so a tile's S buffer is free as soon as the
// softmax has read it: S of the next key tile is computed while the
// exponentials of the current one run, and the two query tiles' softmax
// chains take turns on the tensor cores.
//
// Warp roles (384 threads per CTA):
//   warps 0-3  softmax of tile 0, one thread per row (warp w reads
//              tensor-memory lanes 32w..32w+31)
//   warps 4-7  softmax of tile 1
//   warp 8     TMA loads of this CTA's Q tiles and key half-tiles
//   warp 9     TMA loads of this CTA's value half-tiles
//   warp 10    tensor-memory allocation (both CTAs, together); in the even
//              CTA the issue loop of the S products (one elected lane issues)
//   warp 11    in the even CTA, the issue loop of the P.V products
// Every mbarrier wait is bounded; a wait that runs out raises the abort flag
// of both CTAs and the device error word, the roles leave their loops, work
// in flight is drained, and both CTAs meet at a final cluster barrier before
// tensor memory is released.

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

constexpr float kLazyMax = 1.f;   // log2 of the largest probability taken against a stale maximum
constexpr int kWarpK = 8;
constexpr int kWarpV = 9;
constexpr int kWarpMmaS = 10;    // issues S = Q K^T (and allocates tensor memory)
constexpr int kWarpMmaPV = 11;   // issues O += P V
constexpr int kThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;

// Shared-memory layout of one CTA (D = 128).  Every operand tile is stored in
// 64-column (128-byte) boxes with the 128-byte swizzle.
struct PL {
  static constexpr int kBox = 128 * 64 * 2;             // 128 rows x 64 columns
  static constexpr int kTileBytes = 2 * kBox;           // 128 rows x 128 columns
  static constexpr int kKBox = 64 * 64 * 2;             // 64 keys x 64 columns
  static constexpr int kKStage = 2 * kKBox;             // half of a key tile: 64 keys x 128 columns
  static constexpr int kVStage = kBox;                  // half of a value tile: 128 keys x 64 columns
  static constexpr int KST = 3;
  static constexpr int VST = 2;
  static constexpr int kQ = 0;                          // two query tiles
  static constexpr int kP = kQ + 2 * kTileBytes;        // P of the two tiles (bf16, 128 keys)
  static constexpr int kK = kP + 2 * kTileBytes;
  static constexpr int kV = kK + KST * kKStage;
  static constexpr int kBar = kV + VST * kVStage;
  static constexpr int bQ = 0;
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + KST;
  static constexpr int bVFull = bKEmpty + KST;
  static constexpr int bVEmpty = bVFull + VST;
  static constexpr int bSFull = bVEmpty + VST;          // [2]: per query tile
  static constexpr int bSFree = bSFull + 2;             // [2]
  static constexpr int bPFull = bSFree + 2;             // [2]
  static constexpr int bPVDone = bPFull + 2;            // [2]
  static constexpr int bDrain = bPVDone + 2;            // [2]: per issuing warp
  static constexpr int kNumBars = bDrain + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;     // tensor-memory address, abort flag
  static constexpr int kRange = kMisc + 16;             // (min, max) key position per key tile
  static constexpr int kMaxRanges = 1024;
  static constexpr int kBytes = kRange + kMaxRanges * 8;
  static constexpr int kDynamic = kBytes + 1024;        // room to align the base to 1024
  static_assert(kP % 1024 == 0 && kK % 1024 == 0 && kV % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(kDynamic <= 232448, "shared memory budget");
};

// Tensor-memory columns of query tile h.
__device__ __forceinline__ uint32_t col_O(int hh) { return 256u * static_cast<uint32_t>(hh); }
__device__ __forceinline__ uint32_t col_S(int hh) { return 256u * static_cast<uint32_t>(hh) + 128u; }

// Abort state of a CTA of the pair: its own flag, the peer's flag (cluster
// address) and the device error word.
struct PairAbort {
  volatile int* flag;
  uint32_t peer_flag;
  unsigned int* err;
};

__device__ __forceinline__ void pair_abort(const PairAbort& ab) {
  *ab.flag = 1;
  ptx::st_shared_cluster_u32(ab.peer_flag, 1u);
}

// Bounded wait.  On time-out the abort flags of both CTAs and the device
// error word are raised.
__device__ __noinline__ bool pwait_slow(uint32_t bar, uint32_t parity, PairAbort ab, unsigned int code) {
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*ab.flag) return false;
    if ((n & 255u) == 0) {
      if (*reinterpret_cast<volatile unsigned int*>(ab.err) != 0) {
        pair_abort(ab);
        return false;
      }
      if (ptx::global_timer_ns() - t0 > kWaitTimeoutNs) {
        pair_abort(ab);
        raise_error(ab.err, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PairAbort& ab, unsigned int code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return pwait_slow(bar, parity, ab, code);
}

// Warp-cooperative min and max of count >= 0 positions (INT_MAX / INT_MIN if empty).
__device__ __forceinline__ void warp_minmax(const int32_t* pos, int count, int lane, int& mn, int& mx) {
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

// This CTA's two query tiles (128 rows each) and what the pair agrees on.
struct PairQ {
  int valid[2], mn[2], mx[2];   // rows of each tile inside the shard, their min / max position
  int valid_pair;               // rows of the pair's block inside the shard
  int mx_pair;                  // max position over the pair's block
};

__device__ __forceinline__ PairQ pair_q(const AttnParams& p, int rank, int row0, int pr, int lane) {
  PairQ q;
  const int32_t* base = p.q_pos + static_cast<long long>(rank) * p.n_q;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int start = row0 + pr * 2 * kTile + hh * kTile;
    q.valid[hh] = max(0, min(kTile, p.n_q - start));
    warp_minmax(base + start, q.valid[hh], lane, q.mn[hh], q.mx[hh]);
  }
  q.valid_pair = max(0, min(kPairBlockRows, p.n_q - row0));
  int mn2, mx2;
  warp_minmax(base + row0, q.valid_pair, lane, mn2, mx2);
  q.mx_pair = mx2;
  return q;
}

struct KTile {
  int valid, mn, mx;
  bool skip;   // hidden from every row of the pair
};

// Key tile kt of shard `src` seen by a whole warp: staged ranges, else the
// ranges in global memory, else a reduction of the positions.
__device__ __forceinline__ KTile k_tile(const AttnParams& p, int src, int kt, int ktiles, const PairQ& q,
                                        int lane, const int2* rs) {
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
    warp_minmax(p.k_pos + static_cast<long long>(src) * p.n_k + start, k.valid, lane, k.mn, k.mx);
  }
  k.skip = p.causal ? (k.mn > q.mx_pair) : (q.valid_pair == 0);
  return k;
}

__device__ __forceinline__ int ring_src(int rank, int t, int c) {
  int s = (rank - t) % c;
  return s < 0 ? s + c : s;
}

__device__ __forceinline__ int step_src(const AttnParams& p, int rank, int t) {
  return p.kv_all ? 0 : ring_src(rank, t, p.c);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + PL::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + PL::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PL::kMisc + 4);

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const uint32_t pr = ptx::cluster_ctarank();   // 0: the CTA that issues the pair MMAs
  const bool leader = (pr == 0);
  // the leader's barrier i as a cluster address (for arrivals and TMA bytes
  // from either CTA)
  auto lbar = [&](int i) -> uint32_t { return ptx::mapa_shared(bar(i), 0); };
  const PairAbort ab{abort_flag, ptx::mapa_shared(ptx::smem_u32(const_cast<int*>(abort_flag)), pr ^ 1u), p.err};

  // ---- which problem this pair owns -------------------------------------
  // Blocks start roughly in the order of their linear index; that order runs
  // over (batch, key/value head) outermost, then the query blocks (heaviest
  // first), then the G query heads sharing the key/value head: the pairs in
  // flight together read the keys and values of one head, which stay in L2.
  const long long lin = static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x;
  const long long pq = lin >> 1;                       // pair index; the CTA is lin & 1
  const int hl = static_cast<int>(pq % p.G);
  const long long rest = pq / p.G;
  int yb = static_cast<int>(rest % gridDim.y);
  const int bg = static_cast<int>(rest / gridDim.y);
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int h = g * p.G + hl;
  if (p.block_order != nullptr) yb = p.block_order[yb];
  const int rank = yb / p.q_blocks_per_rank;
  const int row0 = (yb % p.q_blocks_per_rank) * kPairBlockRows;   // local row of the pair's first row
  const int ktiles = (p.n_k + kTile - 1) / kTile;

  // ---- set-up ----------------------------------------------------------
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(PL::bQ), 1);
    for (int s = 0; s < PL::KST; ++s) {
      ptx::mbar_init(bar(PL::bKFull + s), 1);
      ptx::mbar_init(bar(PL::bKEmpty + s), 1);
    }
    for (int s = 0; s < PL::VST; ++s) {
      ptx::mbar_init(bar(PL::bVFull + s), 1);
      ptx::mbar_init(bar(PL::bVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(PL::bSFull + i), 1);
      ptx::mbar_init(bar(PL::bSFree + i), 8);    // one arrival per softmax warp of the tile, both CTAs
      ptx::mbar_init(bar(PL::bPFull + i), 8);
      ptx::mbar_init(bar(PL::bPVDone + i), 1);
      ptx::mbar_init(bar(PL::bDrain + i), 1);
    }
    // A device error left by an earlier block or launch: do no work.
    *abort_flag = (*reinterpret_cast<volatile unsigned int*>(p.err) != 0) ? 1 : 0;
    ptx::fence_mbar_init();
  }
  if (warp == kWarpK && lane == 0) {
    ptx::tma_prefetch_desc(&tm_q);
    ptx::tma_prefetch_desc(&tm_k);
  }
  if (warp == kWarpV && lane == 0) ptx::tma_prefetch_desc(&tm_v);
  if (warp == kWarpMmaS) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  int2* const ranges = reinterpret_cast<int2*>(smem + PL::kRange);
  const int nsteps = p.t_end - p.t_begin;
  const bool staged = static_cast<long long>(nsteps) * ktiles <= PL::kMaxRanges;
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
        warp_minmax(p.k_pos + static_cast<long long>(src) * p.n_k + kt * kTile, min(kTile, p.n_k - kt * kTile),
                    lane, mn, mx);
        if (lane == 0) ranges[i] = make_int2(mn, mx);
      }
    }
  }
  auto step_ranges = [&](int t) -> const int2* { return staged ? ranges + (t - p.t_begin) * ktiles : nullptr; };
  ptx::tc_fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised before either sends to the other
  ptx::cluster_sync_all();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const PairQ qt = pair_q(p, rank, row0, static_cast<int>(pr), lane);

  if (warp == kWarpK || warp == kWarpV) {
    // ===================== TMA producers ================================
    const bool is_k = (warp == kWarpK);
    const CUtensorMap* map = is_k ? &tm_k : &tm_v;
    const int nst = is_k ? PL::KST : PL::VST;
    const int full0 = is_k ? PL::bKFull : PL::bVFull;
    const int empty0 = is_k ? PL::bKEmpty : PL::bVEmpty;
    const uint32_t stage0 = sbase + (is_k ? PL::kK : PL::kV);
    const uint32_t stage_bytes = is_k ? PL::kKStage : PL::kVStage;
    const bool q_issued = is_k && !*abort_flag;
    if (q_issued && lane == 0) {
      // Q rows are read by this pair only: evict first, so that the key and
      // value tiles (read by every block) stay in L2
      const uint64_t pol = ptx::l2_policy_evict_first();
      if (leader) ptx::mbar_arrive_expect_tx(bar(PL::bQ), 4 * PL::kTileBytes);
      for (int hh = 0; hh < 2; ++hh)
        for (int x = 0; x < 2; ++x)
          ptx::tma_load_4d_pair_hint(sbase + PL::kQ + hh * PL::kTileBytes + x * PL::kBox, &tm_q, lbar(PL::bQ),
                                     x * 64, h, rank * p.n_q + row0 + static_cast<int>(pr) * 2 * kTile + hh * kTile,
                                     b, pol);
    }
    uint32_t j = 0;
    bool ok = !*abort_flag;
    for (int t = p.t_begin; t < p.t_end && ok; ++t) {
      const int src = step_src(p, rank, t);
      const int2* rs = step_ranges(t);
      unsigned long long nfull = 0, npart = 0, nskip = 0;
      for (int kt = 0; kt < ktiles; ++kt) {
        const KTile k = k_tile(p, src, kt, ktiles, qt, lane, rs);
        if (is_k && p.work != nullptr) {
          // tile classes of this CTA's two tiles against the key tile
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (qt.valid[hh] == 0) continue;
            if (!p.causal || k.mx <= qt.mn[hh]) ++nfull;
            else if (k.mn > qt.mx[hh]) ++nskip;
            else ++npart;
          }
        }
        if (k.skip) continue;
        if (lane == 0) {
          const int s = static_cast<int>(j % nst);
          const uint32_t n = j / nst;
          if (n > 0) ok = pwait(bar(empty0 + s), (n - 1) & 1u, ab, kErrTimeoutEmpty);
          if (ok) {
            const int krow = (p.kv_by_holder ? rank : src) * p.n_k + kt * kTile;
            if (leader) ptx::mbar_arrive_expect_tx(bar(full0 + s), 2 * stage_bytes);
            if (is_k) {
              // this CTA's 64 keys of the tile, both 64-column boxes
              for (int x = 0; x < 2; ++x)
                ptx::tma_load_4d_pair(stage0 + s * stage_bytes + x * PL::kKBox, map, lbar(full0 + s), x * 64, g,
                                      krow + static_cast<int>(pr) * 64, b);
            } else {
              // this CTA's 64 value columns of all 128 keys
              ptx::tma_load_4d_pair(stage0 + s * stage_bytes, map, lbar(full0 + s), static_cast<int>(pr) * 64, g,
                                    krow, b);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++j;
      }
      if (is_k && p.work != nullptr && ok && lane == 0) {
        ra_work* w = p.work + static_cast<long long>(rank) * p.c + t;
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_full), nfull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_partial), npart);
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_skipped), nskip);
      }
    }
    if (lane == 0 && *abort_flag && leader) {
      // The leader's full barriers count both CTAs' bytes: let the loads in
      // flight land before either CTA leaves (bounded).
      if (q_issued) wait_bar_drain(bar(PL::bQ), 0);
      for (int s = 0; s < nst; ++s) {
        const uint32_t issued = (j > static_cast<uint32_t>(s)) ? (j - 1 - s) / nst + 1 : 0;
        if (issued > 0) wait_bar_drain(bar(full0 + s), (issued - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMmaS || warp == kWarpMmaPV) {
    // ============ pair-MMA issue (even CTA): S and P.V on two warps ============
    // Each issuing warp walks the key tiles in order: S(h, j) as soon as the
    // key half-tiles have landed and both CTAs' softmax of tile h has read
    // S(h, j - 1); P.V(h, j) as soon as both CTAs' P(h, j) is in shared
    // memory.  Neither kind of product waits behind the other.
    if (leader) {
      const bool is_s = (warp == kWarpMmaS);
      constexpr uint32_t idS = ptx::idesc_bf16_f32(256, 128, false);
      constexpr uint32_t idPV = ptx::idesc_bf16_f32(256, D, true);
      bool ok = !is_s || __all_sync(0xffffffffu, pwait(bar(PL::bQ), 0, ab, kErrTimeoutQ));
      bool issued_any = false;
      const uint64_t dQ = ptx::smem_desc_sw128(sbase + PL::kQ, 16, 1024);
      const uint64_t dP = ptx::smem_desc_sw128(sbase + PL::kP, 16, 1024);
      const uint64_t dK = ptx::smem_desc_sw128(sbase + PL::kK, 16, 1024);
      const uint64_t dV = ptx::smem_desc_sw128(sbase + PL::kV, PL::kVStage, 1024);
      uint32_t j = 0;
      for (int t = p.t_begin; t < p.t_end && ok; ++t) {
        const int src = step_src(p, rank, t);
        const int2* rs = step_ranges(t);
        for (int kt = 0; kt < ktiles && ok; ++kt) {
          if (k_tile(p, src, kt, ktiles, qt, lane, rs).skip) continue;
          if (is_s) {
            const int ks = static_cast<int>(j % PL::KST);
            ok = __all_sync(0xffffffffu, pwait(bar(PL::bKFull + ks), (j / PL::KST) & 1u, ab, kErrTimeoutK));
            for (int hh = 0; hh < 2 && ok; ++hh) {
              // S buffer hh is free once both CTAs' softmax read tile j - 1
              if (j >= 1)
                ok = __all_sync(0xffffffffu, pwait(bar(PL::bSFree + hh), (j - 1) & 1u, ab, kErrTimeoutS));
              if (!ok) break;
              ptx::tc_fence_after_sync();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t ao = hh * PL::kTileBytes + (kk / 4) * PL::kBox + (kk % 4) * 32;
                const uint32_t bo = ks * PL::kKStage + (kk / 4) * PL::kKBox + (kk % 4) * 32;
                ptx::tc2_mma_ss_elect(tmem + col_S(hh), dQ + (ao >> 4), dK + (bo >> 4), idS, kk > 0 ? 1u : 0u);
              }
              ptx::tc2_commit_both_elect(bar(PL::bSFull + hh));
              issued_any = true;
            }
            if (ok) ptx::tc2_commit_both_elect(bar(PL::bKEmpty + ks));
          } else {
            const int vs = static_cast<int>(j % PL::VST);
            ok = __all_sync(0xffffffffu, pwait(bar(PL::bVFull + vs), (j / PL::VST) & 1u, ab, kErrTimeoutV));
            for (int hh = 0; hh < 2 && ok; ++hh) {
              ok = __all_sync(0xffffffffu, pwait(bar(PL::bPFull + hh), j & 1u, ab, kErrTimeoutP));
              if (!ok) break;
              ptx::tc_fence_after_sync();
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk) {
                const uint32_t ao = hh * PL::kTileBytes + (kk / 4) * PL::kBox + (kk % 4) * 32;
                ptx::tc2_mma_ss_elect(tmem + col_O(hh), dP + (ao >> 4),
                                      dV + static_cast<uint64_t>((vs * PL::kVStage + kk * 16 * 128) >> 4), idPV, 1u);
              }
              ptx::tc2_commit_both_elect(bar(PL::bPVDone + hh));
              issued_any = true;
            }
            if (ok) ptx::tc2_commit_both_elect(bar(PL::bVEmpty + vs));
          }
          ++j;
        }
      }
      if (!ok && issued_any) {
        // Drain this warp's products before the pair releases its memory.
        const int dr = PL::bDrain + (is_s ? 0 : 1);
        ptx::tc2_commit_both_elect(bar(dr));
        if (!wait_bar_drain(bar(dr), 0)) raise_error(p.err, kErrTimeoutDrain);
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax (both CTAs) ==========================
    const int hh = warp >> 2;                 // query tile of this warpgroup
    const int wq = warp & 3;                  // lane quarter of tensor memory
    const int r = wq * 32 + lane;             // row inside the tile
    const int local_row = row0 + static_cast<int>(pr) * 2 * kTile + hh * kTile + r;
    const bool row_ok = r < qt.valid[hh];
    const long long qrow = static_cast<long long>(rank) * p.n_q + local_row;
    const long long R = static_cast<long long>(p.c) * p.n_q;
    const int qpos = row_ok ? __ldg(p.q_pos + qrow) : INT_MIN;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + col_S(hh);
    const uint32_t tO = tmem + lane_base + col_O(hh);
    // this row of P in shared memory: 128-byte lines of two 64-key boxes,
    // 16-byte chunks permuted by the 128-byte swizzle (chunk ^ row % 8)
    uint8_t* const prow = smem + PL::kP + hh * PL::kTileBytes + r * 128;
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
        const KTile k = k_tile(p, src, kt, ktiles, qt, lane, rs);
        if (k.skip) continue;
        ok = __all_sync(0xffffffffu, pwait(bar(PL::bSFull + hh), j & 1u, ab, kErrTimeoutS));
        if (!ok) break;
        ptx::tc_fence_after_sync();
        const bool masked = (k.valid < kTile) || (p.causal && k.mx > qt.mn[hh]);
        const int32_t* kp = kpos_src + kt * kTile;

        // visibility of each key column (partial tiles only), before S is loaded
        uint32_t bits[4] = {~0u, ~0u, ~0u, ~0u};
        unsigned int nvis = static_cast<unsigned int>(k.valid);
        if (masked && p.k_sorted) {
          // positions increase inside the tile: the visible keys are the prefix
          // of those at or before this row's position.  Equally spaced
          // positions (consecutive, or every c-th in striped shards) give the
          // count directly from the tile's (min, max); otherwise binary search.
          int cnt = k.valid;
          if (p.causal) {
            const int span = k.mx - k.mn;
            if (qpos < k.mn) {
              cnt = 0;
            } else if (span == k.valid - 1) {
              cnt = min(k.valid, qpos - k.mn + 1);
            } else if (p.k_stride > 1 && span == (k.valid - 1) * p.k_stride) {
              cnt = min(k.valid, (qpos - k.mn) / p.k_stride + 1);
            } else {
              cnt = 0;
#pragma unroll
              for (int step = 128; step > 0; step >>= 1)
                if (cnt + step <= k.valid && __ldg(kp + cnt + step - 1) <= qpos) cnt += step;
            }
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
          mx = ptx::fmax3(ptx::fmax3(mc[0], mc[1], mc[2]), ptx::fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
        }
        // S of this tile is in registers: the pair may compute the next key
        // tile's S into the buffer
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lbar(PL::bSFree + hh));

        // The row's reference maximum moves only when the tile's maximum
        // exceeds it by more than kLazyMax (base-2 units): below that the
        // probabilities, taken against the old reference, stay at most
        // 2^kLazyMax, and O and l need no rescaling.
        // Every sum is kept against the same reference, so out = O / l and
        // lse = m + log2 l are unchanged; the first visible key sets it.
        const float m_cand = fmaxf(m_run, mx * sl2);
        const float m_new = (m_cand - m_run > kLazyMax) ? m_cand : m_run;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m_run == m_new) ? 1.f : ptx::ex2(m_run - m_new);
        const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
        const uint64_t negm2 = ptx::f2_pack(-m_use, -m_use);
        uint64_t acc = ptx::f2_pack(0.f, 0.f);
        uint64_t acc1 = ptx::f2_pack(0.f, 0.f);
        // exponentials of 64 keys starting at column c0 -> 32 packed bf16 pairs
        auto exps64 = [&](int c0, uint32_t (&pk)[32]) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint64_t x = ptx::f2_fma(
                ptx::f2_pack(__uint_as_float(sv[c0 + 2 * i]), __uint_as_float(sv[c0 + 2 * i + 1])), sl2x2, negm2);
            float x0, x1;
            ptx::f2_unpack(x, x0, x1);
            const float e0 = ptx::ex2(x0);
            const float e1 = ptx::ex2(x1);
            if (i & 1) acc1 = ptx::f2_add(acc1, ptx::f2_pack(e0, e1));
            else acc = ptx::f2_add(acc, ptx::f2_pack(e0, e1));
            pk[i] = ptx::pack_bf16x2(e0, e1);
          }
        };
        // 64 keys of P into box `box` of this row (eight 16-byte chunks)
        auto store64 = [&](int box, const uint32_t (&pk)[32]) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t off = box * PL::kBox + ((static_cast<uint32_t>(q) ^ (static_cast<uint32_t>(r) & 7u)) << 4);
            *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        };
        {
          uint32_t pk[32];
          exps64(0, pk);
          // P.V of the previous key tile has read P and updated O
          if (j >= 1) ok = __all_sync(0xffffffffu, pwait(bar(PL::bPVDone + hh), (j - 1) & 1u, ab, kErrTimeoutP));
          if (!ok) break;
          store64(0, pk);
        }
        {
          uint32_t pk[32];
          exps64(64, pk);
          store64(1, pk);
        }
        ptx::fence_proxy_async_smem();
        // rescale O when the row maximum rose (P.V of the previous tile is done)
        if (__any_sync(0xffffffffu, (alpha != 1.f) && (m_run != -INFINITY))) {
          ptx::tc_fence_after_sync();
          const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t u[32];
            ptx::tmem_ld32(tO + cc * 32, u);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float y0, y1;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(u[i]), __uint_as_float(u[i + 1])), a2), y0, y1);
              u[i] = __float_as_uint(y0);
              u[i + 1] = __float_as_uint(y1);
            }
            ptx::tmem_st32(tO + cc * 32, u);
          }
          ptx::tmem_wait_st();
        }
        float sm0, sm1;
        ptx::f2_unpack(ptx::f2_add(acc, acc1), sm0, sm1);
        l_run = l_run * alpha + (sm0 + sm1);
        m_run = m_new;
        if (row_ok) pairs += nvis;
        ptx::tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lbar(PL::bPFull + hh));
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
    if (ok && j > 0) ok = __all_sync(0xffffffffu, pwait(bar(PL::bPVDone + hh), (j - 1) & 1u, ab, kErrTimeoutO));
    if (ok) {
      ptx::tc_fence_after_sync();
      if (p.finalize) {
        const int orow = row_ok ? qpos : 0;
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        const long long obase = ((static_cast<long long>(b) * p.S_out + orow) * p.Hq + h) * D;
        // the output is written once and not read here: evict first, so that
        // it does not push the key and value tiles (read by every pair) out
        // of L2
        const uint64_t opol = ptx::l2_policy_evict_first();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          ptx::tmem_ld32(tO + cc * 32, u);
          if (row_ok && p.out_f32) {
            float* d = static_cast<float*>(p.out) + obase + cc * 32;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::st_global_v4_hint(d + 4 * i,
                                     make_uint4(__float_as_uint(__uint_as_float(u[4 * i]) * inv_l),
                                                __float_as_uint(__uint_as_float(u[4 * i + 1]) * inv_l),
                                                __float_as_uint(__uint_as_float(u[4 * i + 2]) * inv_l),
                                                __float_as_uint(__uint_as_float(u[4 * i + 3]) * inv_l)),
                                     opol);
          } else if (row_ok) {
            __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(p.out) + obase + cc * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 0]) * inv_l, __uint_as_float(u[8 * i + 1]) * inv_l);
              w.y = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv_l, __uint_as_float(u[8 * i + 3]) * inv_l);
              w.z = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv_l, __uint_as_float(u[8 * i + 5]) * inv_l);
              w.w = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv_l, __uint_as_float(u[8 * i + 7]) * inv_l);
              ptx::st_global_v4_hint(d + 8 * i, w, opol);
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
  // Neither CTA releases tensor memory (or leaves, taking its shared memory)
  // before the pair's last MMA and load have completed.
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::cluster_sync_all();
  if (warp == kWarpMmaS) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

// Pair kernel (D = 128, bf16): grid x = 2 B Hq (the pairs), y = the 512-row
// query blocks.
int launch_attn_pair(const AttnParams& p, const void* q, const void* k, const void* v, long long q_rows_total,
                     long long k_rows_total, void* stream) {
  if (p.D != 128) return static_cast<int>(cudaErrorInvalidValue);
  CUtensorMap mq, mk, mv;
  std::memset(&mq, 0, sizeof(mq));
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  launch_stage() = "cuTensorMapEncodeTiled";
  int e = make_tma_map_bf16(&mq, q, p.B, q_rows_total, p.Hq, 128, kTile);
  if (!e) e = make_tma_map_bf16(&mk, k, p.B, k_rows_total, p.Hkv, 128, 64);
  if (!e) e = make_tma_map_bf16(&mv, v, p.B, k_rows_total, p.Hkv, 128, kTile);
  if (e) return e;
  const int smem = PL::kDynamic;
  launch_stage() = "cudaFuncSetAttribute (pair kernel)";
  cudaError_t ce = cudaFuncSetAttribute(attn_fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (ce != cudaSuccess) return static_cast<int>(ce);
  const int yb = (p.y_blocks > 0) ? p.y_blocks : p.c * p.q_blocks_per_rank;
  dim3 grid(static_cast<unsigned>(2 * p.B * p.Hq), static_cast<unsigned>(yb));
  launch_stage() = "pair kernel launch";
  attn_fwd_pair_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(mq, mk, mv, p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace ra
