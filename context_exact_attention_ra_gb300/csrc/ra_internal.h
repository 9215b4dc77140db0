// Internal interfaces between the C-ABI layer (ra_api.cpp), the host
// scheduler (ra_sched.cpp) and the CUDA kernels.  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <vector_types.h>

#include "ra.h"

namespace ra {

constexpr int kTile = 128;        // query rows and keys per tile
constexpr int kPairRows = 256;    // query rows per single-CTA tensor-core block (two tiles, D = 64)
constexpr int kPairBlockRows = 512;   // query rows per CTA-pair block (two tiles per CTA, D = 128)
constexpr int kMaxOrderedBlocks = 12288;  // heavy-first ordering limit (48 KB of keys)

// Parameters of one launch of the attention kernels (both the tensor-core
// bf16 kernel and the exact fp32 kernel).  A launch covers `c` problems
// ("ranks"); rank r attends its n_q query rows (rows r*n_q .. of q) to the
// n_k key rows of rank (r - t) mod c for every ring step t in
// [t_begin, t_end).  For a single ra_block_attn call c = 1 and t = 0.
struct AttnParams {
  int B, Hq, Hkv, G, D;
  int c;
  int n_q, n_k;                // rows per rank
  int t_begin, t_end;          // ring steps handled by this launch
  int kv_all;                  // 1: one step over all c*n_k key rows (all-gather), no ring
  int k_sorted;                // 1: key positions increase inside every key tile (the library's
                               //    own layouts), so a row's visible keys in a tile are a prefix
  int kv_by_holder;            // 1: the block held at a step sits in the holder's slot of k, v
                               //    (rows rank*n_k ..), its positions are the source's
  int k_stride;                // > 1: key positions inside a tile may step by this much (striped
                               //    shards: c); a tile whose (min, max) span is (count - 1) * stride
                               //    (or count - 1) holds equally spaced positions
  int q_blocks_per_rank;       // ceil(n_q / rows per block)
  int causal;
  float scale_log2;            // scale * log2(e)

  const int32_t* q_pos;        // [c*n_q]
  const int32_t* k_pos;        // [c*n_k]
  const int2* k_ranges;        // [c*ceil(n_k/128)] (min, max) position per key tile, or nullptr

  const void* q;               // [B, c*n_q, Hq, D]   (fp32 kernel; bf16 uses tensor maps)
  const void* k;               // [B, c*n_k, Hkv, D]
  const void* v;

  // online-softmax state, indexed by q row (c*n_q rows)
  float* o_state;              // [B, c*n_q, Hq, D]
  float* m_state;              // [B, Hq, c*n_q]
  float* l_state;
  int load_state;              // read (o, m, l) before the first step
  int store_state;             // write (o, m, l) after the last step
  // normalised output (finalize): row = q_pos[q row] of an S_out-row tensor
  int finalize;
  int out_f32;                 // output element type: 1 = float32, 0 = the input dtype
  void* out;                   // [B, S_out, Hq, D]
  float* lse;                  // [B, Hq, S_out] or nullptr
  int S_out;

  ra_work* work;               // [c*c] (rank*c + step) or nullptr
  unsigned int* err;           // device error word
  const int32_t* block_order;  // [c*q_blocks_per_rank] or nullptr
  int y_blocks;                // blocks along grid y; 0: c * q_blocks_per_rank (all of them)
};

// Parameters of the decode (split-K over shards) kernels.
struct DecodeParams {
  int B, R, S, n, c, layout, Hq, Hkv, D, causal;
  float scale_log2;
  const void* q;               // [B, R, Hq, D] bf16, the new tokens' queries
  const int32_t* q_pos;        // [R] their global positions
  const void* k;               // [B, S, Hkv, D] bf16, natural order
  const void* v;
  int P;                       // partials per query row (blocks over the shards' 128-key tiles)
  float* part_o;               // [P, B, R, Hq, D]
  float* part_m;               // [P, B, Hq, R] (base-2 units)
  float* part_l;
  void* out;                   // [B, R, Hq, D]
  int out_f32;
  float* lse;                  // [B, Hq, R] or nullptr
  unsigned int* err;           // device error word (bounded waits that ran out)
};

// Error bits written into the device error word.
enum : unsigned int {
  kErrTimeoutQ = 1u << 0,
  kErrTimeoutK = 1u << 1,
  kErrTimeoutV = 1u << 2,
  kErrTimeoutS = 1u << 3,
  kErrTimeoutP = 1u << 4,
  kErrTimeoutO = 1u << 5,
  kErrTimeoutDrain = 1u << 6,
  kErrTimeoutEmpty = 1u << 7,
  kErrSelfTest = 1u << 8,       // the self-test's deliberately unsatisfied wait
};

// ---- launchers (return a cudaError_t as int; 0 = success) -------------
// Tensor map over a [B][rows][H][D] bf16 tensor: boxes of 64 columns x 1 head x
// box_rows rows, 128-byte swizzle (ra_tma.cpp).  Returns a cudaError_t value.
int make_tma_map_bf16(CUtensorMap* map, const void* base, int B, long long rows, int H, int D,
                      int box_rows);
// The keys of striped shard r (rows r, r + c, ...) as a 5-D view {D, H, c, S / c, B}.
int make_tma_map_bf16_strided(CUtensorMap* map, const void* base, int B, long long S, int H, int D, int c,
                              int box_rows);
int launch_attn_tc(const AttnParams& p, const void* q, const void* k, const void* v,
                   long long q_rows_total, long long k_rows_total, void* stream);
// The same on clusters of two CTAs (pair MMAs), D = 128 (attn_pair_sm103.cu).
int launch_attn_pair(const AttnParams& p, const void* q, const void* k, const void* v,
                     long long q_rows_total, long long k_rows_total, void* stream);
int launch_attn_f32(const AttnParams& p, void* stream);
int launch_state_init(int B, int rows, int Hq, int D, float* o, float* m, float* l, void* stream);
int launch_pack(const void* q, const void* k, const void* v, int B, int S, int Hq, int Hkv,
                int D, int elem_bytes, int c, int layout, void* qp, void* kp, void* vp,
                int32_t* pos, void* stream);
int launch_tile_ranges(const int32_t* pos, int c, int n, int2* ranges, void* stream);
// Heavy-first block order; per_rank: each rank's blocks ordered among
// themselves (rank r's list at order[r * blocks_per_rank]).
int launch_block_order(const int32_t* pos, int c, int n, int rows_per_block,
                       int blocks_per_rank, int32_t* order, void* stream, int per_rank = 0);
struct MergeArgs {
  int P;
  const float* outs[RA_MERGE_MAX_PARTIALS];
  const float* ms[RA_MERGE_MAX_PARTIALS];
  const float* ls[RA_MERGE_MAX_PARTIALS];
};
int launch_merge(const MergeArgs& a, int B, int S, int Hq, int D, int out_dtype, void* out,
                 float* lse, const int32_t* out_row, int S_out, void* stream);
int launch_zero(void* ptr, size_t bytes, void* stream);
int launch_decode(const DecodeParams& p, void* stream);
// The tensor-core decode (decode_tc_sm103.cu): D = 64 or 128, every layout
// (each contiguous stretch of a shard tiled on its own, striped shards through
// a strided view).
bool decode_tc_applies(int D, int n, int layout);
int decode_tc_partials(int B, int Hkv, int G, int R, int n, int c, int layout);
int launch_decode_tc(const DecodeParams& p, void* stream);
// The device error word of the current device (its CUDA context), looked up
// on first use in that context.  Two words after it the kernels find the
// device address of the host mirror (or null), which they set when they raise
// an error; `mirror` (may be null) receives the host view of that mirror.
unsigned int* device_error_word(int* cuda_err, volatile unsigned int** mirror = nullptr);
// A unique, nonzero identity of the calling thread's current CUDA context, or
// 0 when there is none yet (caches of per-device handles are keyed by it, so
// that a device reset, which ends the context, never leaves a stale handle).
unsigned long long current_context_id();
// Name of the host step that produced the last launcher error (thread-local).
const char*& launch_stage();
// Wait for `stream`, read the device error word into *value and, when
// `clear`, clear it and its host mirror.  Returns a cudaError_t value.
int read_and_clear_error(void* stream, unsigned int* value, bool clear = true);
int launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, void* stream);

// ---- host scheduler (ra_sched.cpp) ------------------------------------
void shard_positions(int S, int c, int layout, int32_t* pos);
void expected_work(int S, int c, int layout, int causal, ra_work* out);

}  // namespace ra
