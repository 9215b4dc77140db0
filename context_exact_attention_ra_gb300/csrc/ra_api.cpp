// C ABI of the ring-attention library: argument checks, workspace layout,
// and the order of launches.  Every check runs on the host before anything
// is launched.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "ra.h"
#include "ra_internal.h"

namespace {
// NVTX range for profilers (a no-op unless a tool is attached).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};
// Name of ring step t for the per-step ranges (the tool reads it during the push).
const char* step_name(int t) {
  thread_local char name[32];
  std::snprintf(name, sizeof(name), "ring step %d", t);
  return name;
}
}  // namespace

namespace {

using ra::AttnParams;

constexpr double kLn2 = 0.69314718055994530942;
constexpr double kLog2e = 1.44269504088896340736;
constexpr size_t kAlign = 256;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_bytes(int dtype) { return dtype == RA_F32 ? 4 : 2; }

thread_local char g_last_error[320] = "";

// Record a failed CUDA call (where, error name, code, text) for ra_last_error().
ra_status cuda_fail(int e, const char* where) {
  const cudaError_t ce = static_cast<cudaError_t>(e);
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d): %s", where, cudaGetErrorName(ce),
                e, cudaGetErrorString(ce));
  return RA_ERR_CUDA;
}

ra_status cuda_status(int e) { return e == 0 ? RA_OK : cuda_fail(e, ra::launch_stage()); }

ra_status check_shape(const ra_shape& s) {
  if (s.B < 0 || s.Sq < 0 || s.Sk < 0 || s.Hq <= 0 || s.Hkv <= 0) return RA_ERR_INVALID;
  if (s.Hq % s.Hkv != 0) return RA_ERR_INVALID;
  if (s.dtype != RA_BF16 && s.dtype != RA_F32) return RA_ERR_UNSUPPORTED;
  if (s.D != 64 && s.D != 128) return RA_ERR_UNSUPPORTED;
  if (!std::isfinite(s.scale) || !(s.scale > 0.f)) return RA_ERR_INVALID;
  // Index arithmetic in the kernels is 64-bit; grid x holds 2*B*Hq (CTA pairs).
  if (static_cast<long long>(s.B) * s.Hq > 0x3fffffffLL) return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

ra_status check_ring(const ra_shape& s, int c, int layout) {
  ra_status st = check_shape(s);
  if (st != RA_OK) return st;
  if (s.Sq != s.Sk) return RA_ERR_INVALID;
  if (c < 1) return RA_ERR_INVALID;
  if (layout != RA_CONTIGUOUS && layout != RA_ZIGZAG && layout != RA_STRIPED) return RA_ERR_INVALID;
  const long long S = s.Sq;
  if ((layout == RA_CONTIGUOUS || layout == RA_STRIPED) && S % c != 0) return RA_ERR_INVALID;
  if (layout == RA_ZIGZAG && S % (2LL * c) != 0) return RA_ERR_INVALID;
  return RA_OK;
}

bool mode_ok(int mode) {
  return mode == RA_MODE_FUSED || mode == RA_MODE_PER_STEP || mode == RA_MODE_ALLGATHER;
}

// Output element type: the input dtype, or float32 (the fp32 result before
// rounding; for f32 inputs the two coincide).
bool out_dtype_ok(const ra_shape& s, int out_dtype) {
  return out_dtype == s.dtype || out_dtype == RA_F32;
}

// Query rows per thread block of the attention kernel the shape runs on: the
// CTA-pair kernel (bf16, D = 128), the single-CTA tensor-core kernel (bf16,
// D = 64) or the exact fp32 kernel.
int rows_per_block(const ra_shape& s) {
  if (s.dtype != RA_BF16) return ra::kTile;
  return s.D == 128 ? ra::kPairBlockRows : ra::kPairRows;
}

int blocks_per_rank(const ra_shape& s, int n_q) {
  const int rpb = rows_per_block(s);
  return (n_q + rpb - 1) / rpb;
}

// Regions of a ring workspace, as byte offsets from its base.
struct RingWs {
  size_t qp, kp, vp, pos, ranges, order, work, o, m, l, total;
};

RingWs ring_ws(const ra_shape& s, int c, int mode) {
  RingWs w;
  const size_t eb = static_cast<size_t>(elem_bytes(s.dtype));
  const size_t S = static_cast<size_t>(s.Sq), B = static_cast<size_t>(s.B);
  const size_t D = static_cast<size_t>(s.D);
  const int n = c > 0 ? s.Sq / c : 0;
  const size_t nblocks = static_cast<size_t>(c) * blocks_per_rank(s, n);
  size_t off = 0;
  w.qp = off;    off = round_up(off + B * S * s.Hq * D * eb);
  w.kp = off;    off = round_up(off + B * S * s.Hkv * D * eb);
  w.vp = off;    off = round_up(off + B * S * s.Hkv * D * eb);
  w.pos = off;   off = round_up(off + S * sizeof(int32_t));
  w.ranges = off;
  off = round_up(off + static_cast<size_t>(c) * ((n + ra::kTile - 1) / ra::kTile) * 2 * sizeof(int32_t));
  w.order = off; off = round_up(off + nblocks * sizeof(int32_t));
  w.work = off;  off = round_up(off + static_cast<size_t>(c) * c * sizeof(ra_work));
  if (mode == RA_MODE_PER_STEP) {
    w.o = off;   off = round_up(off + B * S * s.Hq * D * sizeof(float));
    w.m = off;   off = round_up(off + B * s.Hq * S * sizeof(float));
    w.l = off;   off = round_up(off + B * s.Hq * S * sizeof(float));
  } else {
    w.o = w.m = w.l = 0;
  }
  w.total = off;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

AttnParams base_params(const ra_shape& s, int c, int n_q, int n_k, int causal) {
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.Hq / s.Hkv;
  p.D = s.D;
  p.c = c;
  p.n_q = n_q;
  p.n_k = n_k;
  p.q_blocks_per_rank = blocks_per_rank(s, n_q);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(s.scale) * kLog2e);
  return p;
}

// The device error word of the current device for the kernels.  A bounded
// wait that ran out earlier on this device, and has not yet been read with
// ra_device_error(), is seen here through the word's host mirror (a plain
// host read, no synchronisation) and refuses the call with RA_ERR_TIMEOUT:
// kernels launched while the word is set would return without computing.
ra_status error_word_or_refuse(unsigned int** ew) {
  int err = 0;
  volatile unsigned int* mirror = nullptr;
  *ew = ra::device_error_word(&err, &mirror);
  if (*ew == nullptr) return cuda_fail(err, "device error word lookup");
  if (mirror != nullptr && *mirror != 0u) {
    std::snprintf(g_last_error, sizeof(g_last_error),
                  "a device wait timed out earlier on this device and is still pending; "
                  "ra_device_error() reads and clears it");
    return RA_ERR_TIMEOUT;
  }
  return RA_OK;
}

ra_status launch_attn(const AttnParams& p, const ra_shape& s, long long q_rows, long long k_rows,
                      void* stream) {
  if (static_cast<long long>(p.c) * p.q_blocks_per_rank > 65535) return RA_ERR_UNSUPPORTED;
  ra::launch_stage() = "kernel launch";
  int e = (s.dtype == RA_BF16) ? ra::launch_attn_tc(p, p.q, p.k, p.v, q_rows, k_rows, stream)
                               : ra::launch_attn_f32(p, stream);
  return cuda_status(e);
}

}  // namespace

extern "C" {

const char* ra_status_string(int status) {
  switch (status) {
    case RA_OK: return "ok";
    case RA_ERR_INVALID: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported configuration";
    case RA_ERR_CUDA: return "CUDA error";
    case RA_ERR_TIMEOUT: return "device wait timed out";
    case RA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

const char* ra_version(void) { return "ra-gb300 0.1 sm_103a"; }

const char* ra_last_error(void) { return g_last_error; }

ra_status ra_state_init(ra_shape shp, float* o, float* m, float* l, ra_stream_t stream) {
  ra_status st = check_shape(shp);
  if (st != RA_OK) return st;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (o == nullptr || m == nullptr || l == nullptr || !aligned16(o)) return RA_ERR_INVALID;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  return cuda_status(ra::launch_state_init(shp.B, shp.Sq, shp.Hq, shp.D, o, m, l, stream));
}

ra_status ra_block_attn(const void* q, const void* k, const void* v, const int32_t* q_pos,
                        const int32_t* k_pos, int causal, ra_shape shp, float* o, float* m,
                        float* l, ra_work* work, ra_stream_t stream) {
  ra_status st = check_shape(shp);
  if (st != RA_OK) return st;
  if (shp.B == 0 || shp.Sq == 0 || shp.Sk == 0) return RA_OK;
  if (!q || !k || !v || !q_pos || !k_pos || !o || !m || !l) return RA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return RA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(work) & 7u) != 0) return RA_ERR_INVALID;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  AttnParams p = base_params(shp, 1, shp.Sq, shp.Sk, causal);
  p.q_pos = q_pos;
  p.k_pos = k_pos;
  p.q = q;
  p.k = k;
  p.v = v;
  p.t_begin = 0;
  p.t_end = 1;
  p.o_state = o;
  p.m_state = m;
  p.l_state = l;
  p.load_state = 1;
  p.store_state = 1;
  p.finalize = 0;
  p.work = work;
  p.err = ew;
  return launch_attn(p, shp, shp.Sq, shp.Sk, stream);
}

ra_status ra_lse_merge(int P, const float* const* outs, const float* const* ms,
                       const float* const* ls, ra_shape shp, void* out, float* lse,
                       ra_stream_t stream) {
  ra_status st = check_shape(shp);
  if (st != RA_OK) return st;
  if (P < 1 || P > RA_MERGE_MAX_PARTIALS) return RA_ERR_INVALID;
  if (!outs || !ms || !ls) return RA_ERR_INVALID;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (out == nullptr || !aligned16(out)) return RA_ERR_INVALID;
  ra::MergeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.P = P;
  for (int i = 0; i < P; ++i) {
    if (!outs[i] || !ms[i] || !ls[i] || !aligned16(outs[i])) return RA_ERR_INVALID;
    a.outs[i] = outs[i];
    a.ms[i] = ms[i];
    a.ls[i] = ls[i];
  }
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  return cuda_status(ra::launch_merge(a, shp.B, shp.Sq, shp.Hq, shp.D, shp.dtype, out, lse,
                                      nullptr, shp.Sq, stream));
}

size_t ra_ring_forward_workspace_size(ra_shape shp, int c, int layout, int mode) {
  if (check_ring(shp, c, layout) != RA_OK) return 0;
  if (!mode_ok(mode)) return 0;
  return ring_ws(shp, c, mode).total;
}

ra_status ra_ring_prepare(const void* q, const void* k, const void* v, ra_shape shp, int c,
                          int layout, void* workspace, size_t ws_bytes, ra_stream_t stream) {
  const Range range("ra_ring_prepare");
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)) return RA_ERR_INVALID;
  const RingWs w = ring_ws(shp, c, RA_MODE_FUSED);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < w.total)
    return RA_ERR_WORKSPACE;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  int e = ra::launch_pack(q, k, v, shp.B, shp.Sq, shp.Hq, shp.Hkv, shp.D, elem_bytes(shp.dtype),
                          c, layout, at<void>(workspace, w.qp), at<void>(workspace, w.kp),
                          at<void>(workspace, w.vp), at<int32_t>(workspace, w.pos), stream);
  if (e) return cuda_fail(e, ra::launch_stage());
  const int n = shp.Sq / c;
  e = ra::launch_tile_ranges(at<int32_t>(workspace, w.pos), c, n, at<int2>(workspace, w.ranges),
                             stream);
  if (e) return cuda_fail(e, ra::launch_stage());
  // Heavy-first block order (used by causal calls): depends on positions only.
  const int total_blocks = c * blocks_per_rank(shp, n);
  if (total_blocks > 1 && total_blocks <= ra::kMaxOrderedBlocks) {
    e = ra::launch_block_order(at<int32_t>(workspace, w.pos), c, n, rows_per_block(shp),
                               blocks_per_rank(shp, n), at<int32_t>(workspace, w.order), stream);
    if (e) return cuda_fail(e, ra::launch_stage());
  }
  return RA_OK;
}

ra_status ra_ring_attend(ra_shape shp, int c, int layout, int causal, int mode, int out_dtype,
                         void* out, float* lse, void* workspace, size_t ws_bytes, int count_work,
                         ra_stream_t stream) {
  const Range range("ra_ring_attend");
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (!mode_ok(mode)) return RA_ERR_INVALID;
  if (!out_dtype_ok(shp, out_dtype)) return RA_ERR_INVALID;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (out == nullptr || !aligned16(out)) return RA_ERR_INVALID;
  const RingWs w = ring_ws(shp, c, mode);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < w.total)
    return RA_ERR_WORKSPACE;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;

  const int S = shp.Sq;
  const int n = S / c;
  AttnParams p = base_params(shp, c, n, n, causal);
  p.k_sorted = 1;   // shard rows are in increasing position in every layout
  p.k_stride = (layout == RA_STRIPED) ? c : 1;
  p.q_pos = at<int32_t>(workspace, w.pos);
  p.k_pos = p.q_pos;
  p.k_ranges = at<int2>(workspace, w.ranges);
  p.q = at<void>(workspace, w.qp);
  p.k = at<void>(workspace, w.kp);
  p.v = at<void>(workspace, w.vp);
  p.err = ew;
  p.out = out;
  p.out_f32 = (out_dtype == RA_F32) ? 1 : 0;
  p.lse = lse;
  p.S_out = S;
  if (count_work) {
    p.work = at<ra_work>(workspace, w.work);
    int e = ra::launch_zero(p.work, static_cast<size_t>(c) * c * sizeof(ra_work), stream);
    if (e) return cuda_fail(e, ra::launch_stage());
  }
  const int total_blocks = c * p.q_blocks_per_rank;
  if (causal && total_blocks <= ra::kMaxOrderedBlocks && total_blocks > 1)
    p.block_order = at<int32_t>(workspace, w.order);   // written by ra_ring_prepare
  if (mode == RA_MODE_FUSED) {
    p.t_begin = 0;
    p.t_end = c;
    p.finalize = 1;
    return launch_attn(p, shp, S, S, stream);
  }
  if (mode == RA_MODE_ALLGATHER) {
    // one step over the gathered keys: the rank-major buffer holds all c
    // shards in rank order, i.e. exactly what an all-gather delivers
    p.kv_all = 1;
    p.n_k = S;
    p.t_begin = 0;
    p.t_end = 1;
    p.finalize = 1;
    // per-rank key-tile ranges coincide with the gathered buffer's tiles only
    // when shards are whole tiles; otherwise the kernel reduces them itself
    if (n % ra::kTile != 0) {
      p.k_ranges = nullptr;
      p.k_sorted = 0;   // a tile may span two shards
    }
    return launch_attn(p, shp, S, S, stream);
  }
  // Per-step: one launch per ring step, the state carried through the
  // workspace between launches.  The first step starts from the empty state
  // (out = 0, m = -inf, l = 0, set in the kernel rather than read back) and the
  // last one ends with out / l and lse in its epilogue instead of storing the
  // state -- the same arithmetic as the separate finalisation, so the result
  // is bitwise the fused mode's either way.
  p.o_state = at<float>(workspace, w.o);
  p.m_state = at<float>(workspace, w.m);
  p.l_state = at<float>(workspace, w.l);
  for (int t = 0; t < c; ++t) {
    const Range step(step_name(t));
    p.t_begin = t;
    p.t_end = t + 1;
    p.load_state = (t > 0) ? 1 : 0;
    p.store_state = (t + 1 < c) ? 1 : 0;
    p.finalize = (t + 1 < c) ? 0 : 1;
    st = launch_attn(p, shp, S, S, stream);
    if (st != RA_OK) return st;
  }
  return RA_OK;
}

ra_status ra_ring_read_work(ra_shape shp, int c, int layout, int mode, const void* workspace,
                            size_t ws_bytes, ra_work* host_per_rank_step, ra_stream_t stream) {
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (host_per_rank_step == nullptr) return RA_ERR_INVALID;
  const RingWs w = ring_ws(shp, c, mode);
  if (workspace == nullptr || ws_bytes < w.total) return RA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamSynchronize");
  ce = cudaMemcpy(host_per_rank_step, static_cast<const char*>(workspace) + w.work,
                  static_cast<size_t>(c) * c * sizeof(ra_work), cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaMemcpy (work counters)");
  return RA_OK;
}

ra_status ra_selftest_wait_timeout(uint32_t limit_us, int leave_pending, ra_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return RA_ERR_INVALID;
  int err = 0;
  unsigned int* ew = ra::device_error_word(&err);
  if (ew == nullptr) return cuda_fail(err, "device error word lookup");
  unsigned int pending = 0;
  int e = ra::read_and_clear_error(stream, &pending);   // start from a clear word
  if (e) return cuda_fail(e, "device error word read");
  e = ra::launch_selftest_timeout(ew, static_cast<uint64_t>(limit_us) * 1000u, stream);
  if (e) return cuda_fail(e, ra::launch_stage());
  if (!leave_pending) return ra_device_error(stream);
  unsigned int v = 0;
  e = ra::read_and_clear_error(stream, &v, false);
  if (e) return cuda_fail(e, "device error word read");
  if (v) std::snprintf(g_last_error, sizeof(g_last_error), "device wait timed out (error bits 0x%x)", v);
  return v ? RA_ERR_TIMEOUT : RA_OK;
}

ra_status ra_device_error(ra_stream_t stream) {
  unsigned int v = 0;
  int e = ra::read_and_clear_error(stream, &v);
  if (e) return cuda_fail(e, "device error word read");
  if (v) std::snprintf(g_last_error, sizeof(g_last_error), "device wait timed out (error bits 0x%x)", v);
  return v ? RA_ERR_TIMEOUT : RA_OK;
}

ra_status ra_schedule(int c, int32_t* table) {
  if (c < 1 || table == nullptr) return RA_ERR_INVALID;
  for (int t = 0; t < c; ++t)
    for (int i = 0; i < c; ++i) table[static_cast<long long>(t) * c + i] = ((i - t) % c + c) % c;
  return RA_OK;
}

ra_status ra_shard_positions(int S, int c, int layout, int32_t* pos) {
  ra_shape s{1, S, S, 1, 1, 128, RA_BF16, 1.f};
  ra_status st = check_ring(s, c, layout);
  if (st != RA_OK) return st;
  if (pos == nullptr && S > 0) return RA_ERR_INVALID;
  ra::shard_positions(S, c, layout, pos);
  return RA_OK;
}

ra_status ra_work_expected(int S, int c, int layout, int causal, ra_work* out) {
  ra_shape s{1, S, S, 1, 1, 128, RA_BF16, 1.f};
  ra_status st = check_ring(s, c, layout);
  if (st != RA_OK) return st;
  if (out == nullptr) return RA_ERR_INVALID;
  ra::expected_work(S, c, layout, causal, out);
  return RA_OK;
}

ra_status ra_ring_forward(const void* q, const void* k, const void* v, ra_shape shp, int c,
                          int layout, int causal, int mode, int out_dtype, void* out, float* lse,
                          void* workspace, size_t ws_bytes, ra_report* report,
                          ra_stream_t stream) {
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (!mode_ok(mode)) return RA_ERR_INVALID;
  if (!out_dtype_ok(shp, out_dtype)) return RA_ERR_INVALID;
  if (report != nullptr && report->c != c) return RA_ERR_INVALID;
  st = ra_ring_prepare(q, k, v, shp, c, layout, workspace, ws_bytes, stream);
  if (st != RA_OK) return st;
  st = ra_ring_attend(shp, c, layout, causal, mode, out_dtype, out, lse, workspace, ws_bytes,
                      report != nullptr && report->per_rank_step != nullptr, stream);
  if (st != RA_OK || report == nullptr) return st;

  // Report: device counters, host schedule and derived quantities.
  const int S = shp.Sq;
  const int n = c > 0 ? S / c : 0;
  std::vector<ra_work> wk(static_cast<size_t>(c) * c);
  if (report->per_rank_step != nullptr) {
    if (shp.B > 0 && S > 0) {
      st = ra_ring_read_work(shp, c, layout, mode, workspace, ws_bytes, report->per_rank_step,
                             stream);
      if (st != RA_OK) return st;
    } else {
      std::memset(report->per_rank_step, 0, sizeof(ra_work) * c * c);
    }
  }
  st = ra_device_error(stream);
  if (st != RA_OK) return st;
  if (report->schedule != nullptr) ra_schedule(c, report->schedule);
  std::vector<ra_work> exp(static_cast<size_t>(c) * c);
  double tot_pairs = 0, max_pairs = 0, tot_tiles = 0, max_tiles = 0;
  if (n > 0) {
    ra::expected_work(S, c, layout, causal, exp.data());
    for (int i = 0; i < c; ++i) {
      double pr = 0, tl = 0;
      for (int t = 0; t < c; ++t) {
        const ra_work& e = exp[static_cast<size_t>(i) * c + t];
        pr += static_cast<double>(e.pairs);
        tl += static_cast<double>(e.tiles_full + e.tiles_partial);
      }
      tot_pairs += pr;
      tot_tiles += tl;
      if (pr > max_pairs) max_pairs = pr;
      if (tl > max_tiles) max_tiles = tl;
    }
  }
  report->imbalance_pairs = tot_pairs > 0 ? max_pairs / (tot_pairs / c) : 1.0;
  report->imbalance_tiles = tot_tiles > 0 ? max_tiles / (tot_tiles / c) : 1.0;
  const uint64_t kvb = static_cast<uint64_t>(S) * shp.Hkv * shp.D * 2 *
                       static_cast<uint64_t>(elem_bytes(shp.dtype)) * shp.B;
  report->ring_kv_bytes = kvb;
  report->ring_kv_bytes_sent = kvb / c * (c - 1);
  report->algorithmic_flop = static_cast<uint64_t>(4.0 * shp.B * shp.Hq * shp.D * tot_pairs);
  return RA_OK;
}

namespace {
// Partials of a decode call: one per block over the shards' 128-key tiles.
struct DecodeWs {
  int P;
  size_t o, m, l, total;
};

DecodeWs decode_ws(const ra_shape& s, int c, int layout) {
  DecodeWs w;
  const int n = s.Sk / c;
  w.P = ra::decode_tc_partials(s.B, s.Hkv, s.Hq / s.Hkv, s.Sq, n, c, layout);
  const size_t P = static_cast<size_t>(w.P), B = static_cast<size_t>(s.B), R = static_cast<size_t>(s.Sq);
  size_t off = 0;
  w.o = off;  off = round_up(off + P * B * R * s.Hq * s.D * sizeof(float));
  w.m = off;  off = round_up(off + P * B * s.Hq * R * sizeof(float));
  w.l = off;  off = round_up(off + P * B * s.Hq * R * sizeof(float));
  w.total = off;
  return w;
}

ra_status check_decode(const ra_shape& s, int c, int layout) {
  ra_status st = check_shape(s);
  if (st != RA_OK) return st;
  if (s.dtype != RA_BF16) return RA_ERR_UNSUPPORTED;
  ra_shape ring = s;
  ring.Sq = s.Sk;     // the key sequence must split over c like a ring's
  return check_ring(ring, c, layout);
}
}  // namespace

size_t ra_decode_workspace_size(ra_shape shp, int c, int layout) {
  if (check_decode(shp, c, layout) != RA_OK || shp.Sk == 0) return 0;
  return decode_ws(shp, c, layout).total;
}

ra_status ra_decode_forward(const void* q, const int32_t* q_pos, const void* k, const void* v,
                            ra_shape shp, int c, int layout, int causal, int out_dtype, void* out,
                            float* lse, void* workspace, size_t ws_bytes, ra_stream_t stream) {
  const Range range("ra_decode_forward");
  ra_status st = check_decode(shp, c, layout);
  if (st != RA_OK) return st;
  if (out_dtype != RA_BF16 && out_dtype != RA_F32) return RA_ERR_INVALID;
  if (shp.B == 0 || shp.Sq == 0 || shp.Sk == 0) return RA_OK;
  if (!q || !q_pos || !k || !v || !out) return RA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return RA_ERR_INVALID;
  const DecodeWs w = decode_ws(shp, c, layout);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < w.total)
    return RA_ERR_WORKSPACE;
  if (w.P > 65535) return RA_ERR_UNSUPPORTED;
  ra::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = shp.B;
  p.R = shp.Sq;
  p.S = shp.Sk;
  p.n = shp.Sk / c;
  p.c = c;
  p.layout = layout;
  p.Hq = shp.Hq;
  p.Hkv = shp.Hkv;
  p.D = shp.D;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(shp.scale) * kLog2e);
  p.q = q;
  p.q_pos = q_pos;
  p.k = k;
  p.v = v;
  p.P = w.P;
  p.part_o = at<float>(workspace, w.o);
  p.part_m = at<float>(workspace, w.m);
  p.part_l = at<float>(workspace, w.l);
  p.out = out;
  p.out_f32 = out_dtype == RA_F32 ? 1 : 0;
  p.lse = lse;
  st = error_word_or_refuse(&p.err);
  if (st != RA_OK) return st;
  return cuda_status(ra::launch_decode(p, stream));
}

size_t ra_ring_rotate_workspace_size(ra_shape shp, int c, int layout) {
  if (check_ring(shp, c, layout) != RA_OK) return 0;
  const size_t base = ring_ws(shp, c, RA_MODE_PER_STEP).total;
  const size_t kvb = static_cast<size_t>(shp.B) * shp.Sq * shp.Hkv * shp.D * elem_bytes(shp.dtype);
  return base + 2 * round_up(kvb);
}

ra_status ra_ring_forward_rotate(const void* q, const void* k, const void* v, ra_shape shp,
                                 int c, int layout, int causal, int overlap, int out_dtype,
                                 void* out, float* lse, void* workspace, size_t ws_bytes,
                                 ra_stream_t stream, ra_stream_t copy_stream) {
  const Range range("ra_ring_forward_rotate");
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (!out_dtype_ok(shp, out_dtype)) return RA_ERR_INVALID;
  if (overlap && (copy_stream == nullptr || copy_stream == stream)) return RA_ERR_INVALID;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (out == nullptr || !aligned16(out)) return RA_ERR_INVALID;
  const size_t need = ra_ring_rotate_workspace_size(shp, c, layout);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < need)
    return RA_ERR_WORKSPACE;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  st = ra_ring_prepare(q, k, v, shp, c, layout, workspace, ws_bytes, stream);
  if (st != RA_OK) return st;

  const RingWs w = ring_ws(shp, c, RA_MODE_PER_STEP);
  const int S = shp.Sq, n = S / c;
  const size_t slot_bytes = static_cast<size_t>(n) * shp.Hkv * shp.D * elem_bytes(shp.dtype);
  const size_t batch_bytes = slot_bytes * c;
  const size_t kvb = batch_bytes * shp.B;
  char* kbuf[2] = {at<char>(workspace, w.kp), at<char>(workspace, w.total)};
  char* vbuf[2] = {at<char>(workspace, w.vp), at<char>(workspace, w.total + round_up(kvb))};

  AttnParams p = base_params(shp, c, n, n, causal);
  p.k_sorted = 1;   // shard rows are in increasing position in every layout
  p.k_stride = (layout == RA_STRIPED) ? c : 1;
  p.q_pos = at<int32_t>(workspace, w.pos);
  p.k_pos = p.q_pos;
  p.k_ranges = at<int2>(workspace, w.ranges);
  p.q = at<void>(workspace, w.qp);
  p.err = ew;
  p.kv_by_holder = 1;
  p.o_state = at<float>(workspace, w.o);
  p.m_state = at<float>(workspace, w.m);
  p.l_state = at<float>(workspace, w.l);
  // as in the per-step ring: the first step starts from the empty state, the
  // last one writes out / l and lse from its epilogue
  p.out = out;
  p.out_f32 = (out_dtype == RA_F32) ? 1 : 0;
  p.lse = lse;
  p.S_out = S;
  if (causal && c * p.q_blocks_per_rank <= ra::kMaxOrderedBlocks && c * p.q_blocks_per_rank > 1)
    p.block_order = at<int32_t>(workspace, w.order);

  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStream_t xs = overlap ? static_cast<cudaStream_t>(copy_stream) : cs;
  cudaEvent_t ev_prep = nullptr, ev_copy = nullptr, ev_comp[2] = {nullptr, nullptr};
  cudaError_t ce = cudaEventCreateWithFlags(&ev_prep, cudaEventDisableTiming);
  if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&ev_copy, cudaEventDisableTiming);
  if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&ev_comp[0], cudaEventDisableTiming);
  if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&ev_comp[1], cudaEventDisableTiming);
  if (ce == cudaSuccess && overlap) {
    ce = cudaEventRecord(ev_prep, cs);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(xs, ev_prep, 0);
  }
  for (int t = 0; t < c && ce == cudaSuccess && st == RA_OK; ++t) {
    const Range step(step_name(t));
    if (t > 0 && overlap) ce = cudaStreamWaitEvent(cs, ev_copy, 0);   // block for step t arrived
    if (ce != cudaSuccess) break;
    p.k = kbuf[t & 1];
    p.v = vbuf[t & 1];
    p.t_begin = t;
    p.t_end = t + 1;
    p.load_state = (t > 0) ? 1 : 0;
    p.store_state = (t + 1 < c) ? 1 : 0;
    p.finalize = (t + 1 < c) ? 0 : 1;
    st = launch_attn(p, shp, S, S, stream);
    if (st != RA_OK) break;
    ce = cudaEventRecord(ev_comp[t & 1], cs);
    if (ce != cudaSuccess || t + 1 >= c) continue;
    // SEND to i+1 / RECV from i-1: slot i of the next buffer gets slot i-1 of
    // this one.  It overwrites what step t-1 read, so wait for that step.
    if (overlap && t >= 1) ce = cudaStreamWaitEvent(xs, ev_comp[(t - 1) & 1], 0);
    for (int b = 0; b < shp.B && ce == cudaSuccess; ++b) {
      for (int which = 0; which < 2 && ce == cudaSuccess; ++which) {
        char* src = (which ? vbuf : kbuf)[t & 1] + b * batch_bytes;
        char* dst = (which ? vbuf : kbuf)[(t + 1) & 1] + b * batch_bytes;
        if (c > 1) ce = cudaMemcpyAsync(dst + slot_bytes, src, slot_bytes * (c - 1),
                                        cudaMemcpyDeviceToDevice, xs);
        if (ce == cudaSuccess)
          ce = cudaMemcpyAsync(dst, src + slot_bytes * (c - 1), slot_bytes,
                               cudaMemcpyDeviceToDevice, xs);
      }
    }
    if (ce == cudaSuccess && overlap) ce = cudaEventRecord(ev_copy, xs);
  }
  if (ev_prep) cudaEventDestroy(ev_prep);
  if (ev_copy) cudaEventDestroy(ev_copy);
  if (ev_comp[0]) cudaEventDestroy(ev_comp[0]);
  if (ev_comp[1]) cudaEventDestroy(ev_comp[1]);
  if (ce != cudaSuccess) return cuda_fail(ce, "ring rotation copies");
  return st;
}

size_t ra_ring_forward_hostio_workspace_size(ra_shape shp, int c, int layout, int mode,
                                             int out_dtype) {
  const size_t base = ra_ring_forward_workspace_size(shp, c, layout, mode);
  if (base == 0 || !out_dtype_ok(shp, out_dtype)) return 0;
  const size_t eb = static_cast<size_t>(elem_bytes(shp.dtype));
  const size_t ob = static_cast<size_t>(elem_bytes(out_dtype));
  const size_t S = static_cast<size_t>(shp.Sq), B = static_cast<size_t>(shp.B), D = shp.D;
  return base + round_up(B * S * shp.Hq * D * eb) + 2 * round_up(B * S * shp.Hkv * D * eb) +
         round_up(B * S * shp.Hq * D * ob) + round_up(B * shp.Hq * S * sizeof(float));
}

namespace {
// The device address of pinned host memory that is mapped into the device's
// address space (16-byte aligned), else nullptr.
void* device_view(void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();   // clear the sticky-free error of an unregistered pointer
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  if ((reinterpret_cast<uintptr_t>(a.devicePointer) & 15u) != 0) return nullptr;
  return a.devicePointer;
}
}  // namespace

namespace {
// Streams and events of the pipelined host-buffer ring, created once per
// device (per CUDA context: a device reset ends the context and its streams,
// and the next call creates new ones): a second stream for attention launches,
// one for the Q copies, one for the output copies and a pool of events.  A
// call holds the device's mutex from before the streams are created or the
// pool grows until its last record and wait are enqueued, so host threads that
// share a device take turns, and no thread's event handles move under it.
struct HostioRes {
  std::mutex mu;
  unsigned long long ctx = 0;
  cudaStream_t attn2 = nullptr;
  cudaStream_t copy = nullptr;   // host to device
  cudaStream_t back = nullptr;   // device to host
  std::vector<cudaEvent_t> ev;
};

// The device's resources; the caller locks r->mu and then calls
// hostio_ready(r, nev) before using them.
HostioRes* hostio_res(cudaError_t* ce) {
  static HostioRes res[64];
  int dev = 0;
  *ce = cudaGetDevice(&dev);
  if (*ce != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *ce = cudaErrorInvalidDevice;
    return nullptr;
  }
  return &res[dev];
}

// Creates the streams (first use in this context) and grows the event pool
// to nev; call with r->mu held.
cudaError_t hostio_ready(HostioRes* r, size_t nev) {
  const unsigned long long ctx = ra::current_context_id();
  if (r->attn2 == nullptr || r->ctx != ctx) {
    // handles of an ended context are not destroyed: they died with it
    r->attn2 = r->copy = r->back = nullptr;
    r->ev.clear();
    cudaError_t ce = cudaStreamCreateWithFlags(&r->attn2, cudaStreamNonBlocking);
    if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&r->copy, cudaStreamNonBlocking);
    if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&r->back, cudaStreamNonBlocking);
    if (ce != cudaSuccess) {
      r->attn2 = nullptr;
      return ce;
    }
    r->ctx = ra::current_context_id();
  }
  while (r->ev.size() < nev) {
    cudaEvent_t e;
    cudaError_t ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (ce != cudaSuccess) return ce;
    r->ev.push_back(e);
  }
  return cudaSuccess;
}

// The fused ring with host inputs and outputs, pipelined: K, V and the
// positions are packed first (read over the CPU-GPU link by the pack kernel,
// or copied first when not mapped); each rank's query rows, which are one or
// two contiguous stretches of the natural order per batch in the contiguous
// and zig-zag layouts, are copied by the copy engine on a stream of their own;
// each rank's query blocks then run as a launch of their own, in heavy-first
// order within the rank, as soon as that rank's rows have landed.  Launches
// alternate between the caller's stream and a second one, so that one
// launch's last blocks overlap the next one's first.  The output goes to
// device memory and each rank's rows are copied to out_host on a third stream
// as soon as its launch has finished (cheaper than the epilogue's stores
// crossing the link); lse is written where lse_dst points.
ra_status hostio_pipelined(const void* q_host, const void* k_src, const void* v_src, ra_shape shp,
                           int c, int layout, int causal, int out_dtype, void* out_host, void* dout,
                           float* lse_dst, void* workspace, cudaStream_t s) {
  const RingWs w = ring_ws(shp, c, RA_MODE_FUSED);
  const int S = shp.Sq;
  const int n = S / c;
  const int bpr = blocks_per_rank(shp, n);
  cudaError_t ce = cudaSuccess;
  HostioRes* res = hostio_res(&ce);
  if (res == nullptr) return cuda_fail(ce, "device lookup");
  std::lock_guard<std::mutex> lock(res->mu);
  ce = hostio_ready(res, 2 * static_cast<size_t>(c) + 4);
  if (ce != cudaSuccess) return cuda_fail(ce, "stream / event creation");
  cudaEvent_t e_entry = res->ev[0], e_prep = res->ev[1], e_done2 = res->ev[2], e_back = res->ev[3];
  cudaEvent_t* e_q = res->ev.data() + 4;       // rank r's query rows landed
  cudaEvent_t* e_att = res->ev.data() + 4 + c; // rank r's attention finished
  char* qp = at<char>(workspace, w.qp);
  const char* qh = static_cast<const char*>(q_host);
  const size_t row_bytes = static_cast<size_t>(shp.Hq) * shp.D * elem_bytes(shp.dtype);
  const size_t orow_bytes = static_cast<size_t>(shp.Hq) * shp.D * elem_bytes(out_dtype);
  // Rank r's rows in the natural order, per batch: one stretch (contiguous)
  // or two (zig-zag); `to_packed` also gives their place in the rank-major
  // buffer.  Copies them between dst and src with the given row size.
  auto copy_rank = [&](int r, char* dst, const char* src, size_t rb, bool to_packed,
                       cudaMemcpyKind kind, cudaStream_t st) -> cudaError_t {
    cudaError_t e2 = cudaSuccess;
    for (int b = 0; b < shp.B && e2 == cudaSuccess; ++b) {
      const size_t brow = static_cast<size_t>(b) * S;
      const int parts = (layout == RA_ZIGZAG) ? 2 : 1;
      const size_t len = static_cast<size_t>(n / parts);
      for (int part = 0; part < parts && e2 == cudaSuccess; ++part) {
        const size_t nat = (layout == RA_ZIGZAG) ? static_cast<size_t>(part == 0 ? r : 2 * c - 1 - r) * len
                                                 : static_cast<size_t>(r) * n;
        const size_t pk = static_cast<size_t>(r) * n + part * len;
        const size_t d_row = brow + (to_packed ? pk : nat);
        const size_t s_row = brow + nat;
        e2 = cudaMemcpyAsync(dst + d_row * rb, src + s_row * rb, len * rb, kind, st);
      }
    }
    return e2;
  };

  // Q: rank by rank on the copy stream
  ce = cudaEventRecord(e_entry, s);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(res->copy, e_entry, 0);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(res->back, e_entry, 0);
  for (int r = 0; r < c && ce == cudaSuccess; ++r) {
    ce = copy_rank(r, qp, qh, row_bytes, true, cudaMemcpyHostToDevice, res->copy);
    if (ce == cudaSuccess) ce = cudaEventRecord(e_q[r], res->copy);
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "Q copies");

  // K, V, positions, tile ranges and the per-rank block order on the caller's stream
  int e = ra::launch_pack(nullptr, k_src, v_src, shp.B, S, shp.Hq, shp.Hkv, shp.D, elem_bytes(shp.dtype),
                          c, layout, qp, at<void>(workspace, w.kp), at<void>(workspace, w.vp),
                          at<int32_t>(workspace, w.pos), s);
  if (!e) e = ra::launch_tile_ranges(at<int32_t>(workspace, w.pos), c, n, at<int2>(workspace, w.ranges), s);
  if (!e)
    e = ra::launch_block_order(at<int32_t>(workspace, w.pos), c, n, rows_per_block(shp), bpr,
                               at<int32_t>(workspace, w.order), s, 1);
  if (e) return cuda_fail(e, ra::launch_stage());
  ce = cudaEventRecord(e_prep, s);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(res->attn2, e_prep, 0);
  if (ce != cudaSuccess) return cuda_fail(ce, "event (prepare)");

  int err = 0;
  unsigned int* ew = ra::device_error_word(&err);
  if (ew == nullptr) return cuda_fail(err, "device error word lookup");
  AttnParams p = base_params(shp, c, n, n, causal);
  p.k_sorted = 1;
  p.k_stride = (layout == RA_STRIPED) ? c : 1;
  p.q_pos = at<int32_t>(workspace, w.pos);
  p.k_pos = p.q_pos;
  p.k_ranges = at<int2>(workspace, w.ranges);
  p.q = qp;
  p.k = at<void>(workspace, w.kp);
  p.v = at<void>(workspace, w.vp);
  p.err = ew;
  p.out = dout;
  p.out_f32 = (out_dtype == RA_F32) ? 1 : 0;
  p.lse = lse_dst;
  p.S_out = S;
  p.t_begin = 0;
  p.t_end = c;
  p.finalize = 1;
  p.y_blocks = bpr;
  ra_status st = RA_OK;
  for (int r = 0; r < c && st == RA_OK; ++r) {
    cudaStream_t sr = (r & 1) ? res->attn2 : s;
    ce = cudaStreamWaitEvent(sr, e_q[r], 0);
    if (ce != cudaSuccess) {
      st = cuda_fail(ce, "event (Q rows)");
      break;
    }
    p.block_order = at<int32_t>(workspace, w.order) + static_cast<size_t>(r) * bpr;
    st = launch_attn(p, shp, S, S, sr);
    if (st != RA_OK) break;
    // rank r's output rows back to the host as soon as its launch is done
    ce = cudaEventRecord(e_att[r], sr);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(res->back, e_att[r], 0);
    if (ce == cudaSuccess)
      ce = copy_rank(r, static_cast<char*>(out_host), static_cast<const char*>(dout), orow_bytes, false,
                     cudaMemcpyDeviceToHost, res->back);
    if (ce != cudaSuccess) st = cuda_fail(ce, "output copies");
  }
  // join the other streams back into the caller's, also after an error
  ce = cudaEventRecord(e_done2, res->attn2);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s, e_done2, 0);
  if (ce == cudaSuccess) ce = cudaEventRecord(e_back, res->back);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s, e_back, 0);
  if (st == RA_OK && ce != cudaSuccess) st = cuda_fail(ce, "event (join)");
  return st;
}
}  // namespace

ra_status ra_ring_forward_hostio(const void* q_host, const void* k_host, const void* v_host,
                                 ra_shape shp, int c, int layout, int causal, int mode,
                                 int out_dtype, void* out_host, float* lse_host, void* workspace,
                                 size_t ws_bytes, ra_stream_t stream) {
  ra_status st = check_ring(shp, c, layout);
  if (st != RA_OK) return st;
  if (!mode_ok(mode)) return RA_ERR_INVALID;
  if (!out_dtype_ok(shp, out_dtype)) return RA_ERR_INVALID;
  if (shp.B == 0 || shp.Sq == 0) return RA_OK;
  if (!q_host || !k_host || !v_host || !out_host) return RA_ERR_INVALID;
  const size_t need = ra_ring_forward_hostio_workspace_size(shp, c, layout, mode, out_dtype);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      ws_bytes < need)
    return RA_ERR_WORKSPACE;
  unsigned int* ew = nullptr;
  st = error_word_or_refuse(&ew);
  if (st != RA_OK) return st;
  const size_t base = ra_ring_forward_workspace_size(shp, c, layout, mode);
  const size_t eb = static_cast<size_t>(elem_bytes(shp.dtype));
  const size_t S = static_cast<size_t>(shp.Sq), B = static_cast<size_t>(shp.B), D = shp.D;
  const size_t qb = B * S * shp.Hq * D * eb, kb = B * S * shp.Hkv * D * eb;
  const size_t ob = B * S * shp.Hq * D * static_cast<size_t>(elem_bytes(out_dtype));
  const size_t lb = B * shp.Hq * S * sizeof(float);
  char* p = static_cast<char*>(workspace) + base;
  void* dq = p;  p += round_up(qb);
  void* dk = p;  p += round_up(kb);
  void* dv = p;  p += round_up(kb);
  void* dout = p; p += round_up(ob);
  float* dlse = reinterpret_cast<float*>(p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Outputs: when the host buffers are pinned and mapped into the device's
  // address space, the kernels write them directly (over the CPU-GPU link,
  // while the attention still runs) instead of a copy after the fact.
  void* out_dst = device_view(out_host);
  float* lse_dst = lse_host ? static_cast<float*>(device_view(lse_host)) : nullptr;
  if (out_dst == nullptr) out_dst = dout;
  if (lse_host && lse_dst == nullptr) lse_dst = dlse;
  // Inputs: mapped pinned buffers are read by the shard-pack kernel directly.
  const void* q_src = device_view(const_cast<void*>(q_host));
  const void* k_src = device_view(const_cast<void*>(k_host));
  const void* v_src = device_view(const_cast<void*>(v_host));
  cudaError_t ce = cudaSuccess;
  const int n = static_cast<int>(S) / c;
  const bool pipelined = mode == RA_MODE_FUSED && shp.dtype == RA_BF16 && q_src != nullptr &&
                         out_dst != dout && (layout == RA_CONTIGUOUS || layout == RA_ZIGZAG) &&
                         c * blocks_per_rank(shp, n) <= ra::kMaxOrderedBlocks;
  if (pipelined) {
    if (k_src == nullptr) {
      ce = cudaMemcpyAsync(dk, k_host, kb, cudaMemcpyHostToDevice, s);
      k_src = dk;
    }
    if (ce == cudaSuccess && v_src == nullptr) {
      ce = cudaMemcpyAsync(dv, v_host, kb, cudaMemcpyHostToDevice, s);
      v_src = dv;
    }
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaMemcpyAsync (inputs)");
    st = hostio_pipelined(q_host, k_src, v_src, shp, c, layout, causal, out_dtype, out_host, dout,
                          lse_dst, workspace, s);
    if (st != RA_OK) return st;
    if (lse_host && lse_dst == dlse) ce = cudaMemcpyAsync(lse_host, dlse, lb, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamSynchronize");
    return RA_OK;
  }
  if (q_src == nullptr) {
    ce = cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, s);
    q_src = dq;
  }
  if (ce == cudaSuccess && k_src == nullptr) {
    ce = cudaMemcpyAsync(dk, k_host, kb, cudaMemcpyHostToDevice, s);
    k_src = dk;
  }
  if (ce == cudaSuccess && v_src == nullptr) {
    ce = cudaMemcpyAsync(dv, v_host, kb, cudaMemcpyHostToDevice, s);
    v_src = dv;
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaMemcpyAsync (inputs)");
  st = ra_ring_forward(q_src, k_src, v_src, shp, c, layout, causal, mode, out_dtype, out_dst, lse_dst,
                       workspace, base, nullptr, stream);
  if (st != RA_OK) return st;
  if (out_dst == dout) ce = cudaMemcpyAsync(out_host, dout, ob, cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess && lse_host && lse_dst == dlse)
    ce = cudaMemcpyAsync(lse_host, dlse, lb, cudaMemcpyDeviceToHost, s);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaMemcpyAsync (outputs)");
  ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamSynchronize");
  return RA_OK;
}

}  // extern "C"
