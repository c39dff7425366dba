// Internal declarations shared by the host runtime and the CUDA kernels.
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define OSCAR_HD __host__ __device__
#else
#define OSCAR_HD
#endif

namespace oscar {

constexpr int kDevBadPage = 1;
constexpr int kDevTimeout = 2;
constexpr int kDevBadLen = 4;
constexpr int kDevBadSlot = 8;
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;  // 200 ms per barrier wait

// Size of the file-scope scratch used by the allocation-free decode entry point.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB

// f16 pair (-1.0, -1.0): the pattern into which the decode kernels OR 2-bit codes
constexpr unsigned kCodeMagic = 0xBC00BC00u;

constexpr int kDtypeF32 = 0;
constexpr int kDtypeBF16 = 1;

// Cache geometry (validated copy of oscar_config).
struct Geom {
  int L, Hq, Hkv, D, P, G, S, W, max_req, max_pages_per_req, num_pages;
  int rph;  // 1: one rotation per kv head (R_K, R_V are [Hkv][D][D]); 0: one per layer
  OSCAR_HD int gq() const { return Hq / Hkv; }
  // floats between the rotations of consecutive kv heads (0: every kv head shares one)
  OSCAR_HD size_t rot_stride() const { return rph ? (size_t)D * D : 0; }
  OSCAR_HD size_t row_bytes() const { return (size_t)D / 4; }
  OSCAR_HD size_t sz_bytes() const { return 4 * (size_t)(D / G); }
  OSCAR_HD size_t k_sz_off() const { return (size_t)P * row_bytes(); }
  OSCAR_HD size_t v_codes_off() const { return k_sz_off() + (size_t)P * sz_bytes(); }
  OSCAR_HD size_t v_sz_off() const { return v_codes_off() + (size_t)P * row_bytes(); }
  OSCAR_HD size_t block_bytes() const { return v_sz_off() + (size_t)P * sz_bytes(); }
  OSCAR_HD size_t layer_pool_bytes() const { return (size_t)num_pages * Hkv * block_bytes(); }
  OSCAR_HD size_t pool_bytes() const { return (size_t)L * layer_pool_bytes(); }
  OSCAR_HD int window() const { return S + W; }
  // bf16 elements of one (layer, request slot) window region: [Hkv][2][S+W][D]
  OSCAR_HD size_t slab_req_elems() const { return (size_t)Hkv * 2 * window() * D; }
  OSCAR_HD size_t slab_bytes() const { return (size_t)L * max_req * slab_req_elems() * 2; }
};

// Arguments of the write family (prefill / extend, eviction, append).
struct WriteArgs {
  Geom g;
  int layer;
  const void* K;
  const void* V;
  int dtype;
  const int* cu_seqlens;   // [batch+1] (write) or null (append)
  const int* start_pos;    // [batch] (write) / seq_lens_before (append)
  int batch;
  int total_tokens;
  const float* R_K;
  const float* R_V;
  float clip_K, clip_V;
  const int* block_table;
  int bt_stride;
  const int* req_slot;
  uint8_t* pool;
  uint16_t* slab;
  int* status;
  int hadamard;            // 1: rotation is H_Had . P_br computed by a fast Walsh-Hadamard transform
  int start_offset;        // append: the new token of request b is at start_pos[b] + start_offset
};

// Decode workspace carve-up (offsets in bytes from the workspace base).
struct DecodeWs {
  size_t qfrag_off, qaux_off, qplain_off, part_off, total;
  int max_splits;        // INT2 splits per (request, kv head)
  int pages_per_split;   // multiple of the 4 warps of a split CTA (each warp streams its own pages)
  int nt;                // query n-tiles (max(1, 2*gq/8))
  int win_chunks;        // BF16 window CTAs per (request, kv head): grid.x = win_chunks + max_splits
  int combine_hpc;       // query heads per combine CTA (a power of two dividing Hq, at most 16)
  int combine_jb;        // output channels per combine CTA (32, 64 or 128; divides D)
  int combine_head;      // 1: one CTA per (query head, request) (small batches)
  int combine_part_smem; // 1: the combine CTA stages its split partials in shared memory
  size_t combine_smem;   // dynamic shared memory of the combine kernel
  int fused;             // 1: one launch per decode (query side formed by the split CTAs, last CTA of a
                         //    (request, kv head) merges); no q_rotate or combine kernel
};

struct DecodeArgs {
  Geom g;
  int layer;
  const void* q;
  int q_dtype;
  void* out;
  int out_dtype;
  const int* block_table;
  int bt_stride;
  const int* seq_lens;
  const int* req_slot;
  int batch;
  int max_seq;
  const float* R_K;
  const float* R_V;
  const uint8_t* pool;       // whole pool (all layers)
  const uint16_t* slab;      // whole slab (all layers)
  const uint8_t* bf16_pool;  // comparison kernel: whole BF16 pool
  int* status;
  uint8_t* ws;
  DecodeWs wl;
  int k_exp_K, k_exp_V;      // operand exponents: K (V) scales and zeros enter the f16 MMAs times 2^k
  unsigned code_magic;       // kCodeMagic (f16 pair -1.0, -1.0), a launch argument so it lives in a register
  int defer_tail_page;       // 1: the preceding kernel may still write the last history page (fused step)
  int* tickets;              // one-launch decode: [batch][Hkv] counters, zero between launches (context-owned)
  int pages_before_wait;     // 1: the preceding grid is this chain's own (it waited on everything before it
                             //    and writes no page but, in a fused step, the last history page)
};

// Extend (chunked prefill) attention over the mixed cache.
struct ExtendArgs {
  Geom g;
  int layer;
  const void* q;             // [total_tokens][Hq][D], q_dtype
  int q_dtype;
  const uint16_t* K_new;     // [total_tokens][Hkv][D] bf16: the chunk's own keys and values
  const uint16_t* V_new;
  void* out;                 // [total_tokens][Hq][D], out_dtype
  int out_dtype;
  const int* cu_seqlens;     // [batch + 1]
  const int* prefix_lens;    // [batch]: cached tokens of each request
  int batch;
  int total_tokens;
  int max_chunk;             // host bound on cu_seqlens[b + 1] - cu_seqlens[b] (sizes the grid)
  const int* block_table;
  int bt_stride;
  const int* req_slot;
  const float* R_K;
  const float* R_V;
  const uint8_t* pool;
  const uint16_t* slab;
  int* status;
  uint8_t* ws;               // R_V as f16 hi / lo planes at rvp_off, q' = q R_K [total_tokens][Hq][D] f32 at qrot_off
  size_t rvp_off, qrot_off;
  int k_exp_K, k_exp_V;
  unsigned code_magic;
  // unpacked-prefix form (null: every attention CTA forms its tiles itself): per (request b,
  // kv head h) the pre-pass writes prep_tiles INT2 tiles, prep_wt window tiles and prep_ct
  // chunk tiles, tile j at prep + ((b Hkv + h) (prep_tiles + prep_wt + prep_ct) + j) *
  // extend_prep_tile_bytes(D); a request with more tiles of a kind forms its own
  uint8_t* prep;
  int prep_tiles, prep_wt, prep_ct;
};
size_t extend_workspace_bytes(const Geom& g, long long total_tokens);
size_t extend_prep_tile_bytes(int D);
// INT2 history tiles (64 keys) of a prefix of max_prefix tokens
long long extend_prep_tiles(const Geom& g, long long max_prefix);
// BF16 window tiles of a request, and chunk tiles of a chunk of at most max_chunk tokens
int extend_prep_window_tiles(const Geom& g);
long long extend_prep_chunk_tiles(const Geom& g, long long max_chunk);
void extend_ws_offsets(const Geom& g, size_t* rvp_off, size_t* qrot_off);
int launch_extend(const ExtendArgs& a, void* stream);
// Self-test of the bounded-wait failure path: waits on an mbarrier that nothing arrives on.
int launch_wait_selftest(int* status, long long limit_ns, void* stream);

// Host-side planning (pure functions, no CUDA).
DecodeWs plan_decode(const Geom& g, int batch, int max_seq, bool bf16_pool);
// Operand exponent k for a clip threshold c: c * 2^k < 2^14, so scales
// (<= 2c/3) and zeros (|z| <= c) times 2^k are f16 numbers below 2^14.
// Returns kNoOperandExp when c is outside [2^-86, 2^14).
constexpr int kNoOperandExp = -1000;
int operand_exponent_for_clip(float clip);

// Kernel launchers (return cudaError_t as int).  Each launches on `stream`.
// pdl: a programmatic dependent of the eviction launched just before it
int launch_write(const WriteArgs& a, void* stream, bool pdl);
// Tensor-core (tcgen05) prefill write for BF16 inputs and a dense rotation.
bool write_tc_supported(const WriteArgs& a);
int launch_write_tc(const WriteArgs& a, void* stream, bool pdl);
int launch_evict(const WriteArgs& a, void* stream, bool pdl);
int launch_append(const WriteArgs& a, void* stream, bool pdl);
int launch_q_rotate(const DecodeArgs& a, void* stream, bool pdl);
int launch_decode_splitk(const DecodeArgs& a, void* stream, bool pdl);
int launch_decode_combine(const DecodeArgs& a, void* stream, bool pdl);
// The fused step's first kernel: the query rotation and the append in one grid.
int launch_step_prep(const WriteArgs& w, const DecodeArgs& d, void* stream, bool pdl);
int launch_bf16_prepare(const DecodeArgs& a, void* stream);
// Device address (for the current device) and size of the file-scope decode
// scratch; the first call on a device looks the address up (not during stream
// capture).
int static_decode_scratch(void** out, size_t* capacity);
int launch_bf16_decode(const DecodeArgs& a, void* stream, bool pdl);
int launch_bf16_combine(const DecodeArgs& a, void* stream, bool pdl);

}  // namespace oscar
