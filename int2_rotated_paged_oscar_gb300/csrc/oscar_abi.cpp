// Host runtime and C ABI of the OSCAR INT2 paged KV cache (see include/oscar.h).
//
// Owns: configuration validation, the page allocator (refcounts, free list,
// branch-point prefix forks with copy-on-write of the partial page), decode
// planning (split sizes, workspace carve-up), the device status word, optional
// per-kernel event timing, and the kernel launches on the caller's stream.
// No exception crosses the ABI; errors are status codes plus a thread-local
// message.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/oscar.h"
#include "oscar_internal.h"

using oscar::DecodeArgs;
using oscar::DecodeWs;
using oscar::Geom;
using oscar::WriteArgs;

namespace {

thread_local std::string g_last_error;

oscar_status fail(oscar_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

oscar_status cuda_fail(int err, const char* what) {
  return fail(OSCAR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

struct Timing {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
  double ms = 0.0;
  int launches = 0;
};

}  // namespace

struct oscar_ctx {
  Geom g{};
  uint8_t* pool = nullptr;
  uint16_t* slab = nullptr;
  int* d_status = nullptr;
  int* d_tickets = nullptr;  // one-launch decode counters [max_requests][n_kv_heads], zero between launches
  std::mutex mu;
  std::vector<int32_t> refcount;
  std::vector<int32_t> free_stack;  // top = back
  long long alloc_fail_after = -1;  // fault injection (OSCAR_FAULT_ALLOC_FAIL_AFTER)
  long long allocs_done = 0;
  bool timing = false;
  std::map<std::string, Timing> timers;
  std::vector<cudaEvent_t> event_pool;
  long long launches = 0;
  // per layer: operand exponents of the history's scales and zeros in the
  // decode MMAs (kNoOperandExp until a clip threshold is known for the layer)
  std::vector<int> opexp_K, opexp_V;
  int decode_form = OSCAR_DECODE_AUTO;
};

namespace {

bool is_pow2_in(int v, std::initializer_list<int> allowed) {
  for (int a : allowed)
    if (v == a) return true;
  return false;
}

oscar_status validate(const oscar_config* c, Geom* out) {
  if (!c) return fail(OSCAR_ERR_INVALID, "config is null");
  if (c->num_layers < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->max_requests < 1 ||
      c->max_pages_per_req < 1 || c->num_pages < 1 || c->sink < 0 || c->recent < 1)
    return fail(OSCAR_ERR_INVALID, "config has a non-positive size");
  if (c->n_q_heads % c->n_kv_heads)
    return fail(OSCAR_ERR_UNSUPPORTED, "n_q_heads (%d) is not a multiple of n_kv_heads (%d)", c->n_q_heads,
                c->n_kv_heads);
  const int gq = c->n_q_heads / c->n_kv_heads;
  if (!is_pow2_in(gq, {1, 2, 4, 8})) return fail(OSCAR_ERR_UNSUPPORTED, "GQA ratio %d not in {1,2,4,8}", gq);
  if (!is_pow2_in(c->head_dim, {64, 128})) return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d not in {64,128}", c->head_dim);
  if (!is_pow2_in(c->page_size, {16, 32, 64}))
    return fail(OSCAR_ERR_UNSUPPORTED, "page_size %d not in {16,32,64}", c->page_size);
  if (c->group_size != 32) return fail(OSCAR_ERR_UNSUPPORTED, "group_size %d is not 32", c->group_size);
  if (c->sink + c->recent > 512)
    return fail(OSCAR_ERR_UNSUPPORTED, "sink + recent = %d exceeds 512", c->sink + c->recent);
  if ((long long)c->max_pages_per_req * c->page_size > (1LL << 30))
    return fail(OSCAR_ERR_INVALID, "max_pages_per_req * page_size too large");
  Geom g;
  g.L = c->num_layers;
  g.Hq = c->n_q_heads;
  g.Hkv = c->n_kv_heads;
  g.D = c->head_dim;
  g.P = c->page_size;
  g.G = c->group_size;
  g.S = c->sink;
  g.W = c->recent;
  g.max_req = c->max_requests;
  g.max_pages_per_req = c->max_pages_per_req;
  g.num_pages = c->num_pages;
  if (c->rotation_per_kv_head != 0 && c->rotation_per_kv_head != 1)
    return fail(OSCAR_ERR_INVALID, "rotation_per_kv_head must be 0 or 1");
  g.rph = c->rotation_per_kv_head;
  *out = g;
  return OSCAR_OK;
}

// --------------------------------------------------------------- tracing
cudaEvent_t take_event(oscar_ctx* ctx) {
  if (!ctx->event_pool.empty()) {
    cudaEvent_t e = ctx->event_pool.back();
    ctx->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct LaunchScope {
  oscar_ctx* ctx;
  const char* name;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  // Inside stream capture the two records become external event-record nodes
  // of the graph, so one replay of the graph times the kernel on the device.
  unsigned flags = cudaEventRecordDefault;
  LaunchScope(oscar_ctx* c, const char* n, void* stream) : ctx(c), name(n), s(static_cast<cudaStream_t>(stream)) {
    if (ctx->timing) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        flags = cudaEventRecordExternal;
      a = take_event(ctx);
      b = take_event(ctx);
      if (a) cudaEventRecordWithFlags(a, s, flags);
    }
  }
  void done(int err) {
    if (err == 0) ctx->launches++;
    if (ctx->timing && a && b) {
      cudaEventRecordWithFlags(b, s, flags);
      ctx->timers[name].pending.push_back({a, b});
    }
  }
};

oscar_status need_device(oscar_ctx* ctx) {
  if (!ctx) return fail(OSCAR_ERR_INVALID, "context is null");
  if (!ctx->pool || !ctx->slab || !ctx->d_status)
    return fail(OSCAR_ERR_INVALID, "context was created without device buffers");
  return OSCAR_OK;
}

// The kernels stage R with 16-byte vector loads and bulk copies.
oscar_status check_r_align(const float* R_K, const float* R_V) {
  if ((reinterpret_cast<uintptr_t>(R_K) | reinterpret_cast<uintptr_t>(R_V)) & 15)
    return fail(OSCAR_ERR_INVALID, "R_K and R_V must be 16-byte aligned");
  return OSCAR_OK;
}

oscar_status check_layer(const oscar_ctx* ctx, int32_t layer) {
  if (layer < 0 || layer >= ctx->g.L) return fail(OSCAR_ERR_INVALID, "layer %d out of [0, %d)", layer, ctx->g.L);
  return OSCAR_OK;
}

}  // namespace

// ====================================================================== planning
namespace oscar {

int operand_exponent_for_clip(float clip) {
  if (!(clip > 0.f) || !std::isfinite(clip)) return kNoOperandExp;
  int e2 = 0;
  std::frexp(clip, &e2);  // clip < 2^e2
  const int k = 14 - e2;  // clip * 2^k < 2^14
  return (k < 0 || k > 100) ? kNoOperandExp : k;
}

// Largest batch x n_q_heads that OSCAR_DECODE_AUTO decodes in one launch (query side and
// merge inside the split kernel); 0: the automatic form is always three kernels.
#ifndef OSCAR_FUSED_ROWS_MAX
#define OSCAR_FUSED_ROWS_MAX 0
#endif
constexpr long long kFusedRowsMax = OSCAR_FUSED_ROWS_MAX;

DecodeWs plan_decode(const Geom& g, int batch, int max_seq, bool bf16_pool) {
  DecodeWs w{};
  const int gq = g.Hq / g.Hkv;
  w.nt = gq == 8 ? 2 : 1;
  const int stage_pages = bf16_pool ? 1 : 4;  // INT2: the 4 warps of a split CTA stream pages round-robin
  long long max_pages;
  if (bf16_pool) max_pages = max_seq > 0 ? (max_seq - 1) / g.P + 1 : 0;
  else max_pages = (max_seq - g.W > g.S) ? (long long)(max_seq - g.W - 1) / g.P + 1 : 0;
  const int occ = bf16_pool ? 2 : 3;  // resident CTAs per SM at the kernels' register use
  const long long wave = 152LL * occ;  // resident CTAs of one wave at the kernel's register use
  const long long pairs = (long long)batch * g.Hkv > 0 ? (long long)batch * g.Hkv : 1;
  const long long win_ctas = bf16_pool ? 0 : (long long)batch * g.Hkv * ((g.S + g.W + 15) / 16);
  long long pps = stage_pages;
  if (bf16_pool) {
    // one wave of splits
    long long free_slots = wave < pairs ? pairs : wave;
    long long split_target = free_slots / pairs;
    if (split_target < 1) split_target = 1;
    pps = max_pages > 0 ? (max_pages + split_target - 1) / split_target : stage_pages;
  } else if (max_pages > 0) {
    // INT2: size splits from the step's page count (an upper bound from max_seq).
    // When one wave holds every split, the splits share it with the window CTAs.
    // Otherwise CTAs of at least kMinSplitPages pages run in up to eight waves:
    // the hardware hands each freed slot the next CTA, which evens out ragged
    // lengths, while the partials stay a small fraction of the cache bytes.
    constexpr long long kMinSplitPages = 16;
    const long long total = pairs * max_pages;
    long long ctas = total / kMinSplitPages;
    if (ctas < wave) {
      ctas = wave - win_ctas;
      if (ctas < pairs) ctas = pairs;
    } else if (ctas > 8 * wave) {
      ctas = 8 * wave;
    }
    pps = (total + ctas - 1) / ctas;
  }
  if (pps < stage_pages) pps = stage_pages;
  pps = (pps + stage_pages - 1) / stage_pages * stage_pages;
  // A few long requests whose splits overflow one wave: the last, partial wave costs nearly a
  // whole CTA time, so take the split size (16..48 pages) that minimises waves (rounded up) x
  // (pages + 4), the 4 being a CTA's fixed cost (first-page latency, epilogue) in page times.
  // Batch 1 at 131K: 16 -> 20 pages, 2.4 -> 1.96 waves, 40.6 -> 37.7 us per layer.  Larger
  // batches keep the plan above: their lengths are ragged and their idle splits cost little.
  if (!bf16_pool && max_pages > 0 && batch <= 4 && pairs * max_pages / 16 >= wave) {
    const long long wc = (g.S + g.W + 15) / 16;
    long long best = -1, best_cost = 0;
    for (long long p = 16; p <= 48; p += stage_pages) {
      const long long ctas = ((max_pages + p - 1) / p + wc) * pairs;
      const long long cost = (ctas + wave - 1) / wave * (p + 4);
      if (best < 0 || cost < best_cost) {
        best = p;
        best_cost = cost;
      }
    }
    pps = best;
  }
  long long splits = max_pages > 0 ? (max_pages + pps - 1) / pps : 0;
  while (splits > 1023) {
    pps += stage_pages;
    splits = (max_pages + pps - 1) / pps;
  }
  w.pages_per_split = static_cast<int>(pps);
  w.max_splits = static_cast<int>(splits);
  w.win_chunks = bf16_pool ? 0 : (g.S + g.W + 15) / 16;
  auto align = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  w.qfrag_off = off;
  off = align(off + (size_t)batch * g.Hkv * w.nt * (g.D / 16) * 32 * 8);
  w.qaux_off = off;
  off = align(off + (size_t)batch * g.Hq * 8 * sizeof(float));
  w.qplain_off = off;
  off = align(off + (size_t)batch * g.Hq * g.D * sizeof(float));
  w.part_off = off;
  const size_t slots = (size_t)w.max_splits + (size_t)w.win_chunks;
  off = align(off + (size_t)batch * g.Hq * slots * (g.D + 4) * sizeof(float));
  w.total = off;
  // combine.  Small batches (a CTA per query head covers at most the SMs): one
  // head per CTA with R_V and its partials staged in shared memory.  Otherwise
  // enough CTAs to cover the SMs about twice, each with the fewest redundant
  // merges: widen the output-channel block first (every CTA of a head merges all
  // D rotated channels), then group heads so that one copy of the R_V rows
  // serves several; the partials are staged when the CTA still fits twice on
  // an SM.
  const long long rows = (long long)batch * g.Hq > 0 ? (long long)batch * g.Hq : 1;
  // One launch per decode (the split CTAs form the query side themselves and the
  // last CTA of each (request, kv head) merges its partials): see kFusedRowsMax.
  w.fused = (!bf16_pool && batch <= g.max_req && rows <= kFusedRowsMax) ? 1 : 0;
  const size_t rv_bytes = (size_t)g.D * g.D * sizeof(float);
  const size_t per_head = slots * (g.D + 4) * sizeof(float);
  if (rows <= 152) {
    w.combine_head = 1;
    w.combine_hpc = 1;
    w.combine_jb = g.D;
    w.combine_part_smem = rv_bytes + per_head <= 200 * 1024 ? 1 : 0;
    w.combine_smem = rv_bytes + (w.combine_part_smem ? per_head : 0) + 64;
    return w;
  }
  int jb = 32, hpc = 1;
  auto combine_ctas = [&]() { return rows / hpc * (g.D / jb); };
  while (combine_ctas() > 2 * 152 && jb < g.D) jb *= 2;
  // with a rotation per kv head, the heads of a CTA share one kv head (one R_V)
  const int hpc_max = g.rph ? (gq < 16 ? gq : 16) : 16;
  while (combine_ctas() > 2 * 152 && hpc < hpc_max && g.Hq % (2 * hpc) == 0) hpc *= 2;
  w.combine_head = 0;
  w.combine_hpc = hpc;
  w.combine_jb = jb;
  const size_t base_floats = (size_t)jb * g.D + (size_t)hpc * g.D + (size_t)hpc * jb + 256 + 16;
  const size_t wts_floats = (size_t)hpc * slots;
  const size_t part_floats = (size_t)hpc * slots * (g.D + 4);
  const size_t budget = 110 * 1024;
  w.combine_part_smem = (base_floats + wts_floats + part_floats) * sizeof(float) <= budget ? 1 : 0;
  w.combine_smem = (base_floats + wts_floats + (w.combine_part_smem ? part_floats : 0)) * sizeof(float) + 16;
  return w;
}

}  // namespace oscar

// ====================================================================== C ABI
extern "C" {

const char* oscar_last_error(void) { return g_last_error.c_str(); }

const char* oscar_version(void) { return "oscar-gb300 0.10 (sm_103a)"; }

size_t oscar_int2_pool_bytes(const oscar_config* cfg) {
  Geom g;
  if (validate(cfg, &g) != OSCAR_OK) return 0;
  return g.pool_bytes();
}

size_t oscar_window_slab_bytes(const oscar_config* cfg) {
  Geom g;
  if (validate(cfg, &g) != OSCAR_OK) return 0;
  return g.slab_bytes();
}

size_t oscar_page_block_bytes(const oscar_config* cfg) {
  Geom g;
  if (validate(cfg, &g) != OSCAR_OK) return 0;
  return g.block_bytes();
}

oscar_status oscar_create(const oscar_config* cfg, void* int2_pool, void* window_slab, oscar_ctx** out) {
  if (!out) return fail(OSCAR_ERR_INVALID, "out is null");
  *out = nullptr;
  Geom g;
  oscar_status st = validate(cfg, &g);
  if (st != OSCAR_OK) return st;
  if ((int2_pool == nullptr) != (window_slab == nullptr))
    return fail(OSCAR_ERR_INVALID, "pass both device buffers or neither");
  if (int2_pool && (reinterpret_cast<uintptr_t>(int2_pool) & 15))
    return fail(OSCAR_ERR_INVALID, "int2_pool must be 16-byte aligned");
  if (window_slab && (reinterpret_cast<uintptr_t>(window_slab) & 15))   // 16-byte row loads and bulk copies
    return fail(OSCAR_ERR_INVALID, "window_slab must be 16-byte aligned");
  oscar_ctx* ctx = new (std::nothrow) oscar_ctx();
  if (!ctx) return fail(OSCAR_ERR_OOM, "host allocation failed");
  ctx->g = g;
  ctx->pool = static_cast<uint8_t*>(int2_pool);
  ctx->slab = static_cast<uint16_t*>(window_slab);
  ctx->refcount.assign(g.num_pages, 0);
  ctx->opexp_K.assign(g.L, oscar::kNoOperandExp);
  ctx->opexp_V.assign(g.L, oscar::kNoOperandExp);
  ctx->free_stack.reserve(g.num_pages);
  for (int i = g.num_pages - 1; i >= 0; --i) ctx->free_stack.push_back(i);  // lowest id first
  if (const char* f = std::getenv("OSCAR_FAULT_ALLOC_FAIL_AFTER")) ctx->alloc_fail_after = std::atoll(f);
  if (int2_pool) {
    const size_t tickets = (size_t)g.max_req * g.Hkv * sizeof(int);
    cudaError_t e = cudaMalloc(&ctx->d_status, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(ctx->d_status, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_tickets, tickets);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_tickets, 0, tickets);
    if (e != cudaSuccess) {
      if (ctx->d_status) cudaFree(ctx->d_status);
      if (ctx->d_tickets) cudaFree(ctx->d_tickets);
      delete ctx;
      return cuda_fail(e, "status word and decode counters");
    }
  }
  *out = ctx;
  return OSCAR_OK;
}

oscar_status oscar_destroy(oscar_ctx* ctx) {
  if (!ctx) return OSCAR_OK;
  for (auto& kv : ctx->timers)
    for (auto& p : kv.second.pending) {
      cudaEventDestroy(p.first);
      cudaEventDestroy(p.second);
    }
  for (auto e : ctx->event_pool) cudaEventDestroy(e);
  if (ctx->d_status) cudaFree(ctx->d_status);
  if (ctx->d_tickets) cudaFree(ctx->d_tickets);
  delete ctx;
  return OSCAR_OK;
}

// ---------------------------------------------------------------- allocator
oscar_status oscar_alloc_pages(oscar_ctx* ctx, int32_t n, int32_t* out_ids) {
  if (!ctx || (n > 0 && !out_ids) || n < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_alloc_pages");
  std::lock_guard<std::mutex> lk(ctx->mu);
  if ((size_t)n > ctx->free_stack.size())
    return fail(OSCAR_ERR_OOM, "page pool exhausted: %d requested, %zu free", n, ctx->free_stack.size());
  if (ctx->alloc_fail_after >= 0 && ctx->allocs_done + n > ctx->alloc_fail_after)
    return fail(OSCAR_ERR_OOM, "page allocation failed (fault injection after %lld pages)", ctx->alloc_fail_after);
  for (int i = 0; i < n; ++i) {
    const int32_t id = ctx->free_stack.back();
    ctx->free_stack.pop_back();
    ctx->refcount[id] = 1;
    out_ids[i] = id;
  }
  ctx->allocs_done += n;
  return OSCAR_OK;
}

oscar_status oscar_ref_pages(oscar_ctx* ctx, const int32_t* ids, int32_t n) {
  if (!ctx || (n > 0 && !ids) || n < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_ref_pages");
  std::lock_guard<std::mutex> lk(ctx->mu);
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= ctx->g.num_pages || ctx->refcount[ids[i]] <= 0)
      return fail(OSCAR_ERR_INVALID, "page %d is not allocated", ids[i]);
  for (int i = 0; i < n; ++i) ctx->refcount[ids[i]]++;
  return OSCAR_OK;
}

oscar_status oscar_unref_pages(oscar_ctx* ctx, const int32_t* ids, int32_t n) {
  if (!ctx || (n > 0 && !ids) || n < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_unref_pages");
  std::lock_guard<std::mutex> lk(ctx->mu);
  std::map<int32_t, int> dec;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= ctx->g.num_pages) return fail(OSCAR_ERR_INVALID, "page %d out of range", ids[i]);
    dec[ids[i]]++;
  }
  for (auto& kv : dec)
    if (ctx->refcount[kv.first] < kv.second)
      return fail(OSCAR_ERR_INVALID, "page %d released more often than referenced", kv.first);
  for (auto& kv : dec) {
    ctx->refcount[kv.first] -= kv.second;
    if (ctx->refcount[kv.first] == 0) ctx->free_stack.push_back(kv.first);
  }
  return OSCAR_OK;
}

oscar_status oscar_page_refcount(oscar_ctx* ctx, int32_t id, int32_t* out_refcount) {
  if (!ctx || !out_refcount || id < 0 || id >= ctx->g.num_pages)
    return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_page_refcount");
  std::lock_guard<std::mutex> lk(ctx->mu);
  *out_refcount = ctx->refcount[id];
  return OSCAR_OK;
}

oscar_status oscar_free_page_count(oscar_ctx* ctx, int32_t* out_n) {
  if (!ctx || !out_n) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_free_page_count");
  std::lock_guard<std::mutex> lk(ctx->mu);
  *out_n = static_cast<int32_t>(ctx->free_stack.size());
  return OSCAR_OK;
}

oscar_status oscar_read_pages(oscar_ctx* ctx, int32_t layer, const int32_t* ids, int32_t n, void* host_dst) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  if (n < 0 || (n > 0 && (!ids || !host_dst))) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_read_pages");
  for (int32_t i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= ctx->g.num_pages)
      return fail(OSCAR_ERR_INVALID, "page id %d out of [0, %d)", ids[i], ctx->g.num_pages);
  const size_t bytes = (size_t)ctx->g.Hkv * ctx->g.block_bytes();
  for (int32_t i = 0; i < n; ++i) {
    const uint8_t* src = ctx->pool + ((size_t)layer * ctx->g.num_pages + ids[i]) * bytes;
    const cudaError_t e = cudaMemcpy(static_cast<uint8_t*>(host_dst) + (size_t)i * bytes, src, bytes,
                                     cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read pages");
  }
  return OSCAR_OK;
}

int32_t oscar_pages_needed(const oscar_config* cfg, int32_t seq_len) {
  Geom g;
  if (validate(cfg, &g) != OSCAR_OK || seq_len < 0) return -1;
  const int h_end = seq_len - g.W;
  if (h_end <= g.S) return 0;
  return (h_end - 1) / g.P + 1;
}

oscar_status oscar_fork_prefix(oscar_ctx* ctx, const int32_t* src_bt, int32_t* dst_bt, int32_t n, int32_t src_slot,
                               int32_t dst_slot, void* stream) {
  if (!ctx || !src_bt || !dst_bt) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_fork_prefix");
  const Geom& g = ctx->g;
  if (n < 0 || (long long)n > (long long)g.max_pages_per_req * g.P)
    return fail(OSCAR_ERR_INVALID, "prefix length %d out of range", n);
  if (src_slot < 0 || src_slot >= g.max_req || dst_slot < 0 || dst_slot >= g.max_req || src_slot == dst_slot)
    return fail(OSCAR_ERR_INVALID, "bad request slots %d -> %d", src_slot, dst_slot);
  const int h_end = n - g.W > g.S ? n - g.W : 0;  // history covers [S, h_end)
  const int full = h_end / g.P;
  const bool partial = h_end % g.P != 0;
  for (int i = 0; i < full + (partial ? 1 : 0); ++i)
    if (src_bt[i] < 0 || src_bt[i] >= g.num_pages) return fail(OSCAR_ERR_INVALID, "source page %d unmapped", i);
  int32_t fresh = -1;
  if (partial) {
    oscar_status st = oscar_alloc_pages(ctx, 1, &fresh);
    if (st != OSCAR_OK) return st;
  }
  if (full > 0) {
    oscar_status st = oscar_ref_pages(ctx, src_bt, full);
    if (st != OSCAR_OK) {
      if (partial) oscar_unref_pages(ctx, &fresh, 1);
      return st;
    }
  }
  for (int i = 0; i < g.max_pages_per_req; ++i) dst_bt[i] = -1;
  for (int i = 0; i < full; ++i) dst_bt[i] = src_bt[i];
  if (partial) dst_bt[full] = fresh;
  if (ctx->pool) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t blk = (size_t)g.Hkv * g.block_bytes();
    for (int l = 0; l < g.L; ++l) {
      cudaError_t e = cudaSuccess;
      if (partial)
        e = cudaMemcpyAsync(ctx->pool + l * g.layer_pool_bytes() + (size_t)fresh * blk,
                            ctx->pool + l * g.layer_pool_bytes() + (size_t)src_bt[full] * blk, blk,
                            cudaMemcpyDeviceToDevice, s);
      if (e == cudaSuccess) {
        const size_t req = g.slab_req_elems();
        e = cudaMemcpyAsync(ctx->slab + ((size_t)l * g.max_req + dst_slot) * req,
                            ctx->slab + ((size_t)l * g.max_req + src_slot) * req, req * 2, cudaMemcpyDeviceToDevice, s);
      }
      if (e != cudaSuccess) return cuda_fail(e, "fork copy");
    }
  }
  return OSCAR_OK;
}

// ---------------------------------------------------------------- write path
// Remember the largest clip thresholds a layer's history was written with (as
// the smallest operand exponents); the decode kernels scale the history's BF16
// scales and zeros by 2^k into f16 operands and need |value| * 2^k < 2^14.
static oscar_status record_clip(oscar_ctx* ctx, int32_t layer, float clip_K, float clip_V) {
  if (!(clip_K > 0.f) || !(clip_V > 0.f) || !std::isfinite(clip_K) || !std::isfinite(clip_V))
    return fail(OSCAR_ERR_INVALID, "clip thresholds must be positive and finite");
  const int ek = oscar::operand_exponent_for_clip(clip_K), ev = oscar::operand_exponent_for_clip(clip_V);
  if (ek == oscar::kNoOperandExp || ev == oscar::kNoOperandExp)
    return fail(OSCAR_ERR_UNSUPPORTED, "clip thresholds (%g, %g) outside [2^-86, 16384)", clip_K, clip_V);
  std::lock_guard<std::mutex> lk(ctx->mu);
  int& k = ctx->opexp_K[layer];
  int& v = ctx->opexp_V[layer];
  k = (k == oscar::kNoOperandExp || ek < k) ? ek : k;
  v = (v == oscar::kNoOperandExp || ev < v) ? ev : v;
  return OSCAR_OK;
}

static oscar_status write_common(oscar_ctx* ctx, int32_t layer, const void* K, const void* V, int32_t dtype,
                                 const int32_t* cu_seqlens, const int32_t* start_pos, int32_t batch,
                                 int32_t total_tokens, const float* R_K, const float* R_V, float clip_K,
                                 float clip_V, const int32_t* block_table, int32_t bt_stride, const int32_t* req_slot,
                                 void* stream, int hadamard) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  if (batch < 0 || total_tokens < 0 || bt_stride < 1) return fail(OSCAR_ERR_INVALID, "bad batch/total/bt_stride");
  if (batch == 0) return OSCAR_OK;
  if (!cu_seqlens || !start_pos || !block_table || !req_slot || (total_tokens > 0 && (!K || !V)))
    return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if (!hadamard && (!R_K || !R_V)) return fail(OSCAR_ERR_INVALID, "R_K / R_V are null");
  if (!hadamard && (st = check_r_align(R_K, R_V)) != OSCAR_OK) return st;
  if (dtype != OSCAR_DTYPE_BF16 && dtype != OSCAR_DTYPE_F32) return fail(OSCAR_ERR_INVALID, "bad dtype %d", dtype);
  if ((st = record_clip(ctx, layer, clip_K, clip_V)) != OSCAR_OK) return st;
  WriteArgs a{};
  a.g = ctx->g;
  a.layer = layer;
  a.K = K;
  a.V = V;
  a.dtype = dtype;
  a.cu_seqlens = cu_seqlens;
  a.start_pos = start_pos;
  a.batch = batch;
  a.total_tokens = total_tokens;
  a.R_K = R_K;
  a.R_V = R_V;
  a.clip_K = clip_K;
  a.clip_V = clip_V;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.req_slot = req_slot;
  a.pool = ctx->pool;
  a.slab = ctx->slab;
  a.status = ctx->d_status;
  a.hadamard = hadamard;
  // the write is a programmatic dependent of the eviction (it waits before its first store), so its
  // set-up overlaps the eviction.  The eviction itself follows the previous kernel in full: as a
  // programmatic dependent of a previous write its waiting CTAs held SMs the next write could use
  // (8 x 32K writes 0.346 -> 0.361 ms)
  const bool pdl = !ctx->timing;
  {
    LaunchScope ls(ctx, "evict", stream);
    int e = oscar::launch_evict(a, stream, false);
    ls.done(e);
    if (e) return cuda_fail(e, "evict launch");
  }
  // BF16 rows with a dense rotation: tensor-core kernel; FP32 rows or the Hadamard-only rotation: CUDA cores
  const bool tc = oscar::write_tc_supported(a);
  LaunchScope ls(ctx, tc ? "write_tc" : "write", stream);
  int e = tc ? oscar::launch_write_tc(a, stream, pdl) : oscar::launch_write(a, stream, pdl);
  ls.done(e);
  if (e) return cuda_fail(e, "write launch");
  return OSCAR_OK;
}

oscar_status oscar_write_kv(oscar_ctx* ctx, int32_t layer, const void* K, const void* V, int32_t dtype,
                            const int32_t* cu_seqlens, const int32_t* start_pos, int32_t batch, int32_t total_tokens,
                            const float* R_K, const float* R_V, float clip_K, float clip_V,
                            const int32_t* block_table, int32_t bt_stride, const int32_t* req_slot, void* stream) {
  return write_common(ctx, layer, K, V, dtype, cu_seqlens, start_pos, batch, total_tokens, R_K, R_V, clip_K, clip_V,
                      block_table, bt_stride, req_slot, stream, 0);
}

oscar_status oscar_write_kv_hadamard(oscar_ctx* ctx, int32_t layer, const void* K, const void* V, int32_t dtype,
                                     const int32_t* cu_seqlens, const int32_t* start_pos, int32_t batch,
                                     int32_t total_tokens, float clip_K, float clip_V, const int32_t* block_table,
                                     int32_t bt_stride, const int32_t* req_slot, void* stream) {
  return write_common(ctx, layer, K, V, dtype, cu_seqlens, start_pos, batch, total_tokens, nullptr, nullptr, clip_K,
                      clip_V, block_table, bt_stride, req_slot, stream, 1);
}

static oscar_status prepare_append(oscar_ctx* ctx, int32_t layer, const void* K_new, const void* V_new,
                                   int32_t dtype, const int32_t* seq_lens, int32_t start_offset, int32_t batch,
                                   const float* R_K, const float* R_V, float clip_K, float clip_V,
                                   const int32_t* block_table, int32_t bt_stride, const int32_t* req_slot,
                                   WriteArgs* out) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  if (batch < 0 || bt_stride < 1) return fail(OSCAR_ERR_INVALID, "bad batch/bt_stride");
  if (batch == 0) return OSCAR_OK;
  if (!K_new || !V_new || !seq_lens || !R_K || !R_V || !block_table || !req_slot)
    return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if ((st = check_r_align(R_K, R_V)) != OSCAR_OK) return st;
  if (dtype != OSCAR_DTYPE_BF16 && dtype != OSCAR_DTYPE_F32) return fail(OSCAR_ERR_INVALID, "bad dtype %d", dtype);
  if ((st = record_clip(ctx, layer, clip_K, clip_V)) != OSCAR_OK) return st;
  WriteArgs& a = *out;
  a = WriteArgs{};
  a.g = ctx->g;
  a.layer = layer;
  a.K = K_new;
  a.V = V_new;
  a.dtype = dtype;
  a.start_pos = seq_lens;
  a.start_offset = start_offset;
  a.batch = batch;
  a.R_K = R_K;
  a.R_V = R_V;
  a.clip_K = clip_K;
  a.clip_V = clip_V;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.req_slot = req_slot;
  a.pool = ctx->pool;
  a.slab = ctx->slab;
  a.status = ctx->d_status;
  return OSCAR_OK;
}

oscar_status oscar_append_step(oscar_ctx* ctx, int32_t layer, const void* K_new, const void* V_new, int32_t dtype,
                               const int32_t* seq_lens_before, int32_t batch, const float* R_K, const float* R_V,
                               float clip_K, float clip_V, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, void* stream) {
  WriteArgs a;
  oscar_status st = prepare_append(ctx, layer, K_new, V_new, dtype, seq_lens_before, 0, batch, R_K, R_V, clip_K,
                                   clip_V, block_table, bt_stride, req_slot, &a);
  if (st != OSCAR_OK || batch == 0) return st;
  LaunchScope ls(ctx, "append", stream);
  int e = oscar::launch_append(a, stream, false);
  ls.done(e);
  if (e) return cuda_fail(e, "append launch");
  return OSCAR_OK;
}

oscar_status oscar_set_layer_clip(oscar_ctx* ctx, int32_t layer, float clip_K, float clip_V) {
  if (!ctx) return fail(OSCAR_ERR_INVALID, "ctx is null");
  oscar_status st = check_layer(ctx, layer);
  if (st != OSCAR_OK) return st;
  return record_clip(ctx, layer, clip_K, clip_V);
}

// ---------------------------------------------------------------- decode
oscar_status oscar_decode_workspace_size(const oscar_config* cfg, int32_t batch, int32_t max_seq, size_t* bytes) {
  Geom g;
  oscar_status st = validate(cfg, &g);
  if (st != OSCAR_OK) return st;
  if (!bytes || batch < 0 || max_seq < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to workspace size");
  *bytes = oscar::plan_decode(g, batch, max_seq, false).total;
  return OSCAR_OK;
}

oscar_status oscar_bf16_decode_workspace_size(const oscar_config* cfg, int32_t batch, int32_t max_seq,
                                              size_t* bytes) {
  Geom g;
  oscar_status st = validate(cfg, &g);
  if (st != OSCAR_OK) return st;
  if (!bytes || batch < 0 || max_seq < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to workspace size");
  *bytes = oscar::plan_decode(g, batch, max_seq, true).total;
  return OSCAR_OK;
}

static oscar_status layer_operand_exps(oscar_ctx* ctx, int32_t layer, int* ek, int* ev) {
  std::lock_guard<std::mutex> lk(ctx->mu);
  *ek = ctx->opexp_K[layer];
  *ev = ctx->opexp_V[layer];
  if (*ek == oscar::kNoOperandExp || *ev == oscar::kNoOperandExp)
    return fail(OSCAR_ERR_INVALID,
                "no clip threshold known for layer %d: write to it or call oscar_set_layer_clip first", layer);
  return OSCAR_OK;
}

static oscar_status check_workspace(const void* workspace) {
  if (!workspace) return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(OSCAR_ERR_INVALID, "workspace must be 256-byte aligned");
  return OSCAR_OK;
}

static oscar_status decode_common_checks(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                                         int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                                         const int32_t* seq_lens, int32_t batch, int32_t max_seq) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  if (batch < 0 || bt_stride < 1 || max_seq < 0) return fail(OSCAR_ERR_INVALID, "bad batch/bt_stride/max_seq");
  if ((long long)max_seq > (long long)ctx->g.max_pages_per_req * ctx->g.P)
    return fail(OSCAR_ERR_INVALID, "max_seq %d exceeds max_pages_per_req * page_size", max_seq);
  if (batch == 0) return OSCAR_OK;
  if (!q || !out || !block_table || !seq_lens) return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if (q_dtype != OSCAR_DTYPE_BF16 && q_dtype != OSCAR_DTYPE_F32) return fail(OSCAR_ERR_INVALID, "bad q dtype");
  if (out_dtype != OSCAR_DTYPE_BF16 && out_dtype != OSCAR_DTYPE_F32) return fail(OSCAR_ERR_INVALID, "bad out dtype");
  return OSCAR_OK;
}

// Checks and argument fill shared by every INT2 decode entry point; the
// workspace (caller scratch or the file-scope array) is set by the caller.
static oscar_status prepare_decode_core(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                                        int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                                        const int32_t* seq_lens, const int32_t* req_slot, int32_t batch,
                                        int32_t max_seq, int32_t sink, int32_t recent, const float* R_K,
                                        const float* R_V, DecodeArgs* dst) {
  oscar_status st = decode_common_checks(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens,
                                         batch, max_seq);
  if (st != OSCAR_OK || batch == 0) return st;
  if (sink != ctx->g.S || recent != ctx->g.W)
    return fail(OSCAR_ERR_INVALID, "sink/recent (%d, %d) differ from the cache configuration (%d, %d)", sink, recent,
                ctx->g.S, ctx->g.W);
  if (!req_slot || !R_K || !R_V) return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if ((st = check_r_align(R_K, R_V)) != OSCAR_OK) return st;
  int ek, ev;
  if ((st = layer_operand_exps(ctx, layer, &ek, &ev)) != OSCAR_OK) return st;
  DecodeArgs& a = *dst;
  a = DecodeArgs{};
  a.g = ctx->g;
  a.layer = layer;
  a.k_exp_K = ek;
  a.k_exp_V = ev;
  a.code_magic = oscar::kCodeMagic;
  a.q = q;
  a.q_dtype = q_dtype;
  a.out = out;
  a.out_dtype = out_dtype;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.req_slot = req_slot;
  a.batch = batch;
  a.max_seq = max_seq;
  a.R_K = R_K;
  a.R_V = R_V;
  a.pool = ctx->pool;
  a.slab = ctx->slab;
  a.status = ctx->d_status;
  a.tickets = ctx->d_tickets;
  a.wl = oscar::plan_decode(ctx->g, batch, max_seq, false);
  if (ctx->decode_form == OSCAR_DECODE_THREE_KERNELS) a.wl.fused = 0;
  if (ctx->decode_form == OSCAR_DECODE_ONE_LAUNCH) a.wl.fused = batch <= ctx->g.max_req ? 1 : 0;
  return OSCAR_OK;
}

static oscar_status prepare_decode(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                                   int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, const int32_t* req_slot, int32_t batch, int32_t max_seq,
                                   int32_t sink, int32_t recent, const float* R_K, const float* R_V, void* workspace,
                                   size_t ws_bytes, DecodeArgs* dst) {
  oscar_status st = prepare_decode_core(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens,
                                        req_slot, batch, max_seq, sink, recent, R_K, R_V, dst);
  if (st != OSCAR_OK || batch == 0) return st;
  if ((st = check_workspace(workspace)) != OSCAR_OK) return st;
  dst->ws = static_cast<uint8_t*>(workspace);
  if (ws_bytes < dst->wl.total)
    return fail(OSCAR_ERR_INVALID, "workspace too small: %zu < %zu bytes", ws_bytes, dst->wl.total);
  return OSCAR_OK;
}

// q_rotate (or, in a fused step, step_prep: the rotation and the append in one
// grid), split-K, combine, all as programmatic dependent launches (unless
// kernel timing is on).  The first kernel waits for its predecessor before it
// reads anything that kernel may write, so every later kernel starts with all
// earlier work on the stream complete.  In a fused step split-K reads every
// page except the last history page before its own dependency wait, because
// the append may be writing that page.
static oscar_status launch_decode_chain(oscar_ctx* ctx, DecodeArgs& a, const WriteArgs* append, void* stream) {
  const bool pdl = !ctx->timing;  // timing events between launches would break the programmatic overlap
  a.defer_tail_page = append != nullptr;
  // split-K copies its first pages before its dependency wait only behind a kernel of this
  // chain (q_rotate or step_prep); a one-launch decode follows the caller's last kernel
  a.pages_before_wait = (append != nullptr || !a.wl.fused) ? 1 : 0;
  if (a.wl.fused) {  // one launch (after the append CTAs of a fused step)
    if (append) {
      LaunchScope ls(ctx, "step_prep", stream);
      int e = oscar::launch_step_prep(*append, a, stream, pdl);
      ls.done(e);
      if (e) return cuda_fail(e, "step_prep launch");
    }
    LaunchScope ls(ctx, "decode_splitk", stream);
    int e = oscar::launch_decode_splitk(a, stream, pdl);
    ls.done(e);
    if (e) return cuda_fail(e, "decode_splitk launch");
    return OSCAR_OK;
  }
  if (append) {
    LaunchScope ls(ctx, "step_prep", stream);
    int e = oscar::launch_step_prep(*append, a, stream, pdl);
    ls.done(e);
    if (e) return cuda_fail(e, "step_prep launch");
  } else {
    LaunchScope ls(ctx, "q_rotate", stream);
    int e = oscar::launch_q_rotate(a, stream, pdl);
    ls.done(e);
    if (e) return cuda_fail(e, "q_rotate launch");
  }
  {
    LaunchScope ls(ctx, "decode_splitk", stream);
    int e = oscar::launch_decode_splitk(a, stream, pdl);
    ls.done(e);
    if (e) return cuda_fail(e, "decode_splitk launch");
  }
  LaunchScope ls(ctx, "decode_combine", stream);
  int e = oscar::launch_decode_combine(a, stream, pdl);
  ls.done(e);
  if (e) return cuda_fail(e, "decode_combine launch");
  return OSCAR_OK;
}

oscar_status oscar_decode_attn(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                               int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, const int32_t* req_slot, int32_t batch, int32_t max_seq,
                               int32_t sink, int32_t recent, const float* R_K, const float* R_V, void* workspace,
                               size_t ws_bytes, void* stream) {
  DecodeArgs a;
  oscar_status st = prepare_decode(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens, req_slot,
                                   batch, max_seq, sink, recent, R_K, R_V, workspace, ws_bytes, &a);
  if (st != OSCAR_OK || batch == 0) return st;
  return launch_decode_chain(ctx, a, nullptr, stream);
}

oscar_status oscar_decode_step(oscar_ctx* ctx, int32_t layer, const void* K_new, const void* V_new, int32_t kv_dtype,
                               const void* q, int32_t q_dtype, void* out, int32_t out_dtype,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               const int32_t* req_slot, int32_t batch, int32_t max_seq, int32_t sink, int32_t recent,
                               const float* R_K, const float* R_V, float clip_K, float clip_V, void* workspace,
                               size_t ws_bytes, void* stream) {
  WriteArgs w;
  oscar_status st = prepare_append(ctx, layer, K_new, V_new, kv_dtype, seq_lens, -1, batch, R_K, R_V, clip_K, clip_V,
                                   block_table, bt_stride, req_slot, &w);
  if (st != OSCAR_OK || batch == 0) return st;
  DecodeArgs a;
  st = prepare_decode(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens, req_slot, batch,
                      max_seq, sink, recent, R_K, R_V, workspace, ws_bytes, &a);
  if (st != OSCAR_OK) return st;
  return launch_decode_chain(ctx, a, &w, stream);
}

oscar_status oscar_decode_attn_noalloc(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                                       int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                                       const int32_t* seq_lens, const int32_t* req_slot, int32_t batch,
                                       int32_t max_seq, int32_t sink, int32_t recent, const float* R_K,
                                       const float* R_V, void* stream) {
  // Scratch comes from the library's file-scope device array: nothing here
  // allocates (no cudaMalloc / cudaFree, no torch).
  DecodeArgs a;
  oscar_status st = prepare_decode_core(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens,
                                        req_slot, batch, max_seq, sink, recent, R_K, R_V, &a);
  if (st != OSCAR_OK || batch == 0) return st;
  if (a.wl.total > oscar::kStaticScratchBytes)
    return fail(OSCAR_ERR_INVALID,
                "decode needs %zu bytes of scratch for batch %d, max_seq %d; the allocation-free entry point has "
                "%zu (use oscar_decode_attn with a caller workspace)",
                a.wl.total, batch, max_seq, oscar::kStaticScratchBytes);
  void* scratch = nullptr;
  size_t cap = 0;
  int e = oscar::static_decode_scratch(&scratch, &cap);
  if (e) return cuda_fail(e, "static scratch address");
  a.ws = static_cast<uint8_t*>(scratch);
  return launch_decode_chain(ctx, a, nullptr, stream);
}

// ---------------------------------------------------------------- extend
oscar_status oscar_extend_workspace_size(const oscar_config* cfg, int32_t total_tokens, size_t* bytes) {
  Geom g;
  oscar_status st = validate(cfg, &g);
  if (st != OSCAR_OK) return st;
  if (!bytes || total_tokens < 0) return fail(OSCAR_ERR_INVALID, "bad arguments to extend workspace size");
  *bytes = oscar::extend_workspace_bytes(g, total_tokens);
  return OSCAR_OK;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

oscar_status oscar_extend_workspace_size_unpacked(const oscar_config* cfg, int32_t total_tokens, int32_t batch,
                                                  int32_t max_prefix, int32_t max_chunk, size_t* bytes) {
  Geom g;
  oscar_status st = validate(cfg, &g);
  if (st != OSCAR_OK) return st;
  if (!bytes || total_tokens < 0 || batch < 0 || max_prefix < 0 || max_chunk < 0)
    return fail(OSCAR_ERR_INVALID, "bad arguments to extend workspace size");
  const long long tiles = oscar::extend_prep_tiles(g, max_prefix) + oscar::extend_prep_window_tiles(g) +
                          oscar::extend_prep_chunk_tiles(g, max_chunk);
  *bytes = align256(oscar::extend_workspace_bytes(g, total_tokens)) +
           (size_t)batch * g.Hkv * (size_t)tiles * oscar::extend_prep_tile_bytes(g.D);
  return OSCAR_OK;
}

oscar_status oscar_extend_attn(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, const void* K_new,
                               const void* V_new, int32_t kv_dtype, void* out, int32_t out_dtype,
                               const int32_t* cu_seqlens, const int32_t* prefix_lens, int32_t batch,
                               int32_t total_tokens, int32_t max_chunk, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, const float* R_K, const float* R_V, void* workspace,
                               size_t ws_bytes, void* stream) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  if (batch < 0 || total_tokens < 0 || max_chunk < 0 || bt_stride < 1)
    return fail(OSCAR_ERR_INVALID, "bad batch/total_tokens/max_chunk/bt_stride");
  if (batch == 0 || total_tokens == 0) return OSCAR_OK;
  if (batch > 65535) return fail(OSCAR_ERR_UNSUPPORTED, "extend: batch %d above 65535 (one grid dimension)", batch);
  if (!q || !K_new || !V_new || !out || !cu_seqlens || !prefix_lens || !block_table || !req_slot || !R_K || !R_V ||
      !workspace)
    return fail(OSCAR_ERR_INVALID, "null tensor argument");
  if (kv_dtype != OSCAR_DTYPE_BF16) return fail(OSCAR_ERR_UNSUPPORTED, "extend: K_new / V_new must be BF16");
  if (q_dtype != OSCAR_DTYPE_BF16) return fail(OSCAR_ERR_UNSUPPORTED, "extend: q must be BF16");
  if (out_dtype != OSCAR_DTYPE_BF16 && out_dtype != OSCAR_DTYPE_F32) return fail(OSCAR_ERR_INVALID, "bad out dtype");
  if (128 % ctx->g.gq() != 0)
    return fail(OSCAR_ERR_UNSUPPORTED, "extend: n_q_heads / n_kv_heads = %d must divide 128", ctx->g.gq());
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(OSCAR_ERR_INVALID, "workspace must be 256-byte aligned");
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(K_new) | reinterpret_cast<uintptr_t>(V_new) |
        reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return fail(OSCAR_ERR_INVALID, "q, K_new, V_new and out must be 16-byte aligned");
  if ((st = check_r_align(R_K, R_V)) != OSCAR_OK) return st;
  const size_t need = oscar::extend_workspace_bytes(ctx->g, total_tokens);
  if (ws_bytes < need) return fail(OSCAR_ERR_INVALID, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  int ek, ev;
  if ((st = layer_operand_exps(ctx, layer, &ek, &ev)) != OSCAR_OK) return st;
  oscar::ExtendArgs a{};
  a.g = ctx->g;
  a.layer = layer;
  a.q = q;
  a.q_dtype = q_dtype;
  a.K_new = static_cast<const uint16_t*>(K_new);
  a.V_new = static_cast<const uint16_t*>(V_new);
  a.out = out;
  a.out_dtype = out_dtype;
  a.cu_seqlens = cu_seqlens;
  a.prefix_lens = prefix_lens;
  a.batch = batch;
  a.total_tokens = total_tokens;
  a.max_chunk = max_chunk;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.req_slot = req_slot;
  a.R_K = R_K;
  a.R_V = R_V;
  a.pool = ctx->pool;
  a.slab = ctx->slab;
  a.status = ctx->d_status;
  a.ws = static_cast<uint8_t*>(workspace);
  oscar::extend_ws_offsets(ctx->g, &a.rvp_off, &a.qrot_off);
  a.k_exp_K = ek;
  a.k_exp_V = ev;
  a.code_magic = oscar::kCodeMagic;
  // unpacked-prefix form when the workspace holds, past the base, the window and chunk tiles
  // of every (request, kv head): then as many INT2 tiles per pair as fit, at most what the
  // longest prefix can have
  a.prep = nullptr;
  a.prep_tiles = a.prep_wt = a.prep_ct = 0;
  {
    const size_t base = align256(need);
    const size_t per_tile = (size_t)batch * ctx->g.Hkv * oscar::extend_prep_tile_bytes(ctx->g.D);
    const long long fixed = oscar::extend_prep_window_tiles(ctx->g) + oscar::extend_prep_chunk_tiles(ctx->g, max_chunk);
    if (ws_bytes >= base && (long long)((ws_bytes - base) / per_tile) >= fixed) {
      long long tiles = (long long)((ws_bytes - base) / per_tile) - fixed;
      const long long cap = oscar::extend_prep_tiles(ctx->g, (long long)ctx->g.max_pages_per_req * ctx->g.P);
      if (tiles > cap) tiles = cap;
      a.prep = a.ws + base;
      a.prep_tiles = (int)tiles;
      a.prep_wt = oscar::extend_prep_window_tiles(ctx->g);
      a.prep_ct = (int)oscar::extend_prep_chunk_tiles(ctx->g, max_chunk);
    }
  }
  LaunchScope ls(ctx, "extend", stream);
  int e = oscar::launch_extend(a, stream);
  ls.done(e);
  if (e) return cuda_fail(e, "extend launch");
  return OSCAR_OK;
}

oscar_status oscar_selftest_wait_timeout(oscar_ctx* ctx, int32_t limit_us, void* stream) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if (limit_us < 1 || limit_us > 1000000) return fail(OSCAR_ERR_INVALID, "limit_us %d outside [1, 1e6]", limit_us);
  LaunchScope ls(ctx, "selftest", stream);
  int e = oscar::launch_wait_selftest(ctx->d_status, (long long)limit_us * 1000, stream);
  ls.done(e);
  if (e) return cuda_fail(e, "self-test launch");
  return OSCAR_OK;
}

oscar_status oscar_extend_step(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, const void* K_new,
                               const void* V_new, int32_t kv_dtype, void* out, int32_t out_dtype,
                               const int32_t* cu_seqlens, const int32_t* prefix_lens, int32_t batch,
                               int32_t total_tokens, int32_t max_chunk, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, const float* R_K, const float* R_V, float clip_K,
                               float clip_V, void* workspace, size_t ws_bytes, void* stream) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  if ((st = check_layer(ctx, layer)) != OSCAR_OK) return st;
  // the chunk's write declares these clips anyway; declaring them first lets the first chunk of a
  // fresh layer attend (its prefix is empty, so nothing was written with another clip)
  if ((st = record_clip(ctx, layer, clip_K, clip_V)) != OSCAR_OK) return st;
  st = oscar_extend_attn(ctx, layer, q, q_dtype, K_new, V_new, kv_dtype, out, out_dtype, cu_seqlens, prefix_lens,
                         batch, total_tokens, max_chunk, block_table, bt_stride, req_slot, R_K, R_V, workspace,
                         ws_bytes, stream);
  if (st != OSCAR_OK || batch == 0 || total_tokens == 0) return st;
  return oscar_write_kv(ctx, layer, K_new, V_new, kv_dtype, cu_seqlens, prefix_lens, batch, total_tokens, R_K, R_V,
                        clip_K, clip_V, block_table, bt_stride, req_slot, stream);
}

oscar_status oscar_bf16_decode_attn(oscar_ctx* ctx, int32_t layer, const void* bf16_pool, const void* q,
                                    int32_t q_dtype, void* out, int32_t out_dtype, const int32_t* block_table,
                                    int32_t bt_stride, const int32_t* seq_lens, int32_t batch, int32_t max_seq,
                                    void* workspace, size_t ws_bytes, void* stream) {
  oscar_status st = decode_common_checks(ctx, layer, q, q_dtype, out, out_dtype, block_table, bt_stride, seq_lens,
                                         batch, max_seq);
  if (st != OSCAR_OK || batch == 0) return st;
  if ((st = check_workspace(workspace)) != OSCAR_OK) return st;
  if (!bf16_pool) return fail(OSCAR_ERR_INVALID, "bf16_pool is null");
  if (reinterpret_cast<uintptr_t>(bf16_pool) & 15) return fail(OSCAR_ERR_INVALID, "bf16_pool must be 16-byte aligned");
  if (ctx->g.P != 64) return fail(OSCAR_ERR_UNSUPPORTED, "the BF16 comparison kernel needs page_size 64");
  DecodeArgs a{};
  a.g = ctx->g;
  a.layer = layer;
  a.q = q;
  a.q_dtype = q_dtype;
  a.out = out;
  a.out_dtype = out_dtype;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq = max_seq;
  a.bf16_pool = static_cast<const uint8_t*>(bf16_pool);
  a.status = ctx->d_status;
  a.ws = static_cast<uint8_t*>(workspace);
  a.wl = oscar::plan_decode(ctx->g, batch, max_seq, true);
  if (ws_bytes < a.wl.total)
    return fail(OSCAR_ERR_INVALID, "workspace too small: %zu < %zu bytes", ws_bytes, a.wl.total);
  const bool pdl = !ctx->timing;
  {
    LaunchScope ls(ctx, "bf16_prepare", stream);
    int e = oscar::launch_bf16_prepare(a, stream);
    ls.done(e);
    if (e) return cuda_fail(e, "bf16_prepare launch");
  }
  {
    LaunchScope ls(ctx, "bf16_decode", stream);
    int e = oscar::launch_bf16_decode(a, stream, pdl);
    ls.done(e);
    if (e) return cuda_fail(e, "bf16_decode launch");
  }
  LaunchScope ls(ctx, "bf16_combine", stream);
  int e = oscar::launch_bf16_combine(a, stream, pdl);
  ls.done(e);
  if (e) return cuda_fail(e, "bf16_combine launch");
  return OSCAR_OK;
}

// ---------------------------------------------------------------- status, tracing
oscar_status oscar_check_status(oscar_ctx* ctx, void* stream, int32_t* out_bits) {
  oscar_status st = need_device(ctx);
  if (st != OSCAR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int bits = 0;
  e = cudaMemcpy(&bits, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (out_bits) *out_bits = bits;
  if (bits) {
    cudaMemset(ctx->d_status, 0, sizeof(int));
    // a launch that failed may have left the one-launch decode counters mid-count
    cudaMemset(ctx->d_tickets, 0, (size_t)ctx->g.max_req * ctx->g.Hkv * sizeof(int));
    return fail(OSCAR_ERR_DEVICE, "device status 0x%x (%s%s%s)", bits, (bits & oscar::kDevBadPage) ? "bad page " : "",
                (bits & oscar::kDevTimeout) ? "wait timeout " : "", (bits & oscar::kDevBadLen) ? "bad length " : "");
  }
  return OSCAR_OK;
}

oscar_status oscar_set_decode_form(oscar_ctx* ctx, int32_t form) {
  if (!ctx) return fail(OSCAR_ERR_INVALID, "context is null");
  if (form != OSCAR_DECODE_AUTO && form != OSCAR_DECODE_THREE_KERNELS && form != OSCAR_DECODE_ONE_LAUNCH)
    return fail(OSCAR_ERR_INVALID, "unknown decode form %d", form);
  std::lock_guard<std::mutex> lk(ctx->mu);
  ctx->decode_form = form;
  return OSCAR_OK;
}

oscar_status oscar_set_timing(oscar_ctx* ctx, int32_t enable) {
  if (!ctx) return fail(OSCAR_ERR_INVALID, "context is null");
  ctx->timing = enable != 0;
  return OSCAR_OK;
}

oscar_status oscar_kernel_time(oscar_ctx* ctx, const char* name, double* out_ms, int32_t* out_launches) {
  if (!ctx || !name || !out_ms || !out_launches) return fail(OSCAR_ERR_INVALID, "bad arguments to oscar_kernel_time");
  Timing& t = ctx->timers[name];
  for (auto& p : t.pending) {
    cudaError_t e = cudaEventSynchronize(p.second);
    if (e != cudaSuccess) return cuda_fail(e, "event synchronize");
    float ms = 0.f;
    cudaEventElapsedTime(&ms, p.first, p.second);
    t.ms += ms;
    t.launches++;
    ctx->event_pool.push_back(p.first);
    ctx->event_pool.push_back(p.second);
  }
  t.pending.clear();
  *out_ms = t.ms;
  *out_launches = t.launches;
  return OSCAR_OK;
}

oscar_status oscar_reset_timing(oscar_ctx* ctx) {
  if (!ctx) return fail(OSCAR_ERR_INVALID, "context is null");
  for (auto& kv : ctx->timers) {
    for (auto& p : kv.second.pending) {
      cudaEventSynchronize(p.second);
      ctx->event_pool.push_back(p.first);
      ctx->event_pool.push_back(p.second);
    }
    kv.second.pending.clear();
    kv.second.ms = 0.0;
    kv.second.launches = 0;
  }
  return OSCAR_OK;
}

int64_t oscar_launch_count(oscar_ctx* ctx) { return ctx ? ctx->launches : 0; }

}  // extern "C"
