// Fused decode attention over the mixed-precision paged cache (INT2 history +
// BF16 sink/recent window).
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- the serving
// kernel unpacks, dequantises and inverse-rotates the INT2 history and computes
// attention over it, compatible with paged attention and prefix caching, with
// no extra memory traffic; arXiv abstract -- fused decode kernel, batch-1
// decode faster than BF16 by cutting KV memory traffic.
//
// Formulation (exact rearrangement of softmax(q K^T/sqrt(d)) V over
// K = [Y_K R_K^T ; K_win], V = [Y_V R_V^T ; V_win]):
//   q' = q R_K once per step;  history score_t = q'.y_K,t / sqrt(d);
//   history values accumulate in the rotated basis, acc_rot = sum_t p_t y_V,t;
//   o = (sum_win p v + acc_rot R_V^T) / l, R_V^T applied once per output row.
//
// Kernels (one decode step):
//   q_rotate       q' = q R_K per (request, kv head, channel group); writes the
//                  query-side MMA fragments (f16 hi/lo of q' times a per-head
//                  power of two), the group sums Q_g and q as float32.
//   decode_splitk  grid (window chunks + INT2 splits, kv heads, requests).  Window
//                  chunk CTAs score 16 BF16 window slots each in float32.  INT2
//                  split CTAs stream pages through per-warp rings and run QK and
//                  PV on the tensor cores (mma.sync m16n8k16, f16 operands with
//                  the BF16 group scales folded in; see the split section).  Each
//                  CTA writes one partial (m, l, acc) per query head.
//   decode_combine merges the partials, applies R_V^T once and divides by l.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {

// Scratch of the allocation-free decode entry point (oscar_decode_attn_noalloc):
// a file-scope device array of kStaticScratchBytes.  Every GPU that loads the
// library holds it until the process exits.  Host code never uses the symbol
// as an address; it asks the runtime for the device address once per device
// (static_decode_scratch below).
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kWarps = kThreads / 32;
#include "q_rotate.cuh"
#include "decode_window.cuh"

// ------------------------------------------------------------------ q rotate
// grid (Hkv * D/32, B), block 128: CTA (kvh, grp) of request b runs q_rotate_cta
// (q_rotate.cuh).  Launched as a programmatic dependent of whatever preceded it
// on the stream; it lets its own dependents launch after its wait on that grid,
// so every kernel after it still sees all earlier work complete.
template <int D>
__global__ void __launch_bounds__(kThreads) q_rotate_kernel(DecodeArgs a) {
  __shared__ __align__(16) float sm[kQRotSmemFloats<D>()];
  q_rotate_cta<D>(a, blockIdx.x % (D / 32), blockIdx.x / (D / 32), blockIdx.y, sm,
                  q_out_ws(a, blockIdx.x / (D / 32), blockIdx.y));
}

// ------------------------------------------------------------------ in-CTA query side
// One-launch decode: every INT2 split CTA of a (request, kv head) forms that
// pair's query side itself, after the wait on the preceding grid, with the
// definitions q_rotate_cta uses (q' = q R_K for the gq query heads, the group
// sums Q_g, 2^-e_h from ||q_h||_2 and the MMA fragments).  Thread (c4, part)
// accumulates channels 4 c4 .. 4 c4 + 3 of q' over rows [part RPP, part RPP + RPP)
// of R_K (16-byte loads, eight in flight); the parts are added in a fixed order.
// scr: kQSideSmemFloats<D>() floats of shared memory; qf: fragments [NT][D/16][32]
// (columns of absent heads zero); qaux: [gq][8] as in the workspace.  Ends with
// a barrier after which every thread's shared-memory accesses are ordered
// before later bulk copies into scr.
template <int D>
__host__ __device__ constexpr int kQSideParts() { return kThreads / (D / 4); }
template <int D>
__host__ __device__ constexpr int kQSideSmemFloats() { return 8 * D + kQSideParts<D>() * 8 * D + 8; }

template <int D, int NT>
__device__ __forceinline__ void q_side_cta(const DecodeArgs& a, int kvh, int b, float* scr, uint2* qf, float* qaux) {
  constexpr int C4 = D / 4, PARTS = kQSideParts<D>(), RPP = D / PARTS;
  constexpr int GROUPS = D / 32;
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(scr);                  // [8][D]: q
  float (*red)[8][D] = reinterpret_cast<float (*)[8][D]>(scr + 8 * D);   // [PARTS][8][D]; red[0] ends as q'
  float* nrm = scr + 8 * D + PARTS * 8 * D;                              // [8]
  const Geom& g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = g.gq();
  const size_t qbase = ((size_t)b * g.Hq + (size_t)kvh * gq) * D;
  for (int i = tid; i < gq * D; i += kThreads) qs[i / D][i % D] = load_q(a, qbase + i);
  for (int i = tid; i < NT * (D / 16) * 32; i += kThreads) qf[i] = make_uint2(0u, 0u);
  __syncthreads();
  for (int hh = warp; hh < gq; hh += kWarps) {
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss = fmaf(qs[hh][i], qs[hh][i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) nrm[hh] = sqrtf(ss);
  }
  {
    const int c4 = tid % C4, part = tid / C4;
    const float4* Rg = reinterpret_cast<const float4*>(a.R_K + (size_t)kvh * g.rot_stride()) + c4;
    float acc[8][4];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[hh][c] = 0.f;
#pragma unroll 4
    for (int r = 0; r < RPP; ++r) {
      const int i = part * RPP + r;
      const float4 R4 = __ldg(Rg + (size_t)i * C4);
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        if (hh < gq) {
          const float x = qs[hh][i];
          acc[hh][0] = fmaf(x, R4.x, acc[hh][0]);
          acc[hh][1] = fmaf(x, R4.y, acc[hh][1]);
          acc[hh][2] = fmaf(x, R4.z, acc[hh][2]);
          acc[hh][3] = fmaf(x, R4.w, acc[hh][3]);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh)
      if (hh < gq)
        *reinterpret_cast<float4*>(&red[part][hh][4 * c4]) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
  }
  __syncthreads();
  for (int idx = tid; idx < gq * D; idx += kThreads) {
    const int hh = idx / D, j = idx % D;
    float y = red[0][hh][j];
#pragma unroll
    for (int p = 1; p < PARTS; ++p) y += red[p][hh][j];
    red[0][hh][j] = y;
  }
  __syncthreads();
  float (*qr)[D] = red[0];
  for (int pr = warp; pr < gq * GROUPS; pr += kWarps) {   // Q_g: warp per (head, group)
    const int hh = pr / GROUPS, grp = pr % GROUPS;
    float gs = qr[hh][32 * grp + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
    if (lane == 0) qaux[hh * 8 + 1 + grp] = gs;
  }
  for (int idx = tid; idx < gq * GROUPS * 16; idx += kThreads) {
    const int hh = idx / (GROUPS * 16), grp = (idx >> 4) % GROUPS, sub = idx & 15;
    const int e = q_head_exp(nrm[hh]);
    if (grp == 0 && sub == 0) qaux[hh * 8] = ldexpf(1.f, -e);
    q_frag_entry<D>(qr[hh] + 32 * grp, hh, grp, sub, e, gq, qf);
  }
  fence_proxy_async_smem();
  __syncthreads();
}

// ------------------------------------------------------------------ in-kernel combine
// One-launch decode: each CTA of a (request, kv head) takes a ticket after its
// partials are stored (a device-scope fence by every thread, then one atomic);
// the CTA that draws the last ticket of the pair merges the pair's partials for
// its gq query heads and writes their outputs, so no CTA ever waits on another.
// That CTA puts the counter back to zero for the next launch (stream order: the
// next launch takes tickets only after its wait on this grid).
//   1. R_V (this kv head's) is copied into shared memory by one bulk copy;
//   2. warp per head: the reference M over the pair's partials, then lane c4
//      merges channels 4 c4 .. 4 c4 + 3 of every partial (eight partials' loads
//      in flight, L2 loads: the partials were written by other CTAs): window
//      partials into the plain sum, INT2 partials into the rotated sum, and l;
//   3. thread per output channel j (and k half when D = 64): sum_k rot_k R_V[j][k]
//      for every head from float4 rows, each thread starting at its own k so that
//      a phase of 8 threads reads 8 different bank groups; o = (plain + that) / l.
// Shared memory (from offset 0): R_V [D][D], rot [8][D], plain [8][D], l [8], and
// for D = 64 the second k half's sums [8][D].
template <int D>
__host__ __device__ constexpr int kMergeSmemBytes() {
  return (D * D + 16 * D + 8 + (kThreads / D > 1 ? 8 * D : 0)) * 4;
}

template <int D>
__device__ __noinline__ void fused_merge(const DecodeArgs& a, int b, int kvh, uint8_t* smem, uint64_t* bar) {
  constexpr int LPC = D / 4 < 32 ? D / 4 : 32;   // lanes per partial row (float4 each)
  constexpr int SPW = 32 / LPC;                  // partials a warp reads side by side
  constexpr int NPK = kThreads / D;              // k parts per output channel
  const Geom& g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = g.gq();
  const int wc = a.wl.win_chunks;
  const int stride = wc + a.wl.max_splits;
  const int n = a.seq_lens[b];
  const int nsp = seq_len_ok(a, n) ? min(splits_for(a, n), kMaxSplits) : 0;
  const int nslot = wc + nsp;
  float* Rs = reinterpret_cast<float*>(smem);
  float* rot = Rs + D * D;
  float* plain = rot + 8 * D;
  float* Ls = plain + 8 * D;
  float* xr = Ls + 8;
  fence_proxy_async_smem();   // this thread's earlier shared-memory use, before the bulk copy
  __syncthreads();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, D * D * sizeof(float));
    bulk_g2s(Rs, a.R_V + (size_t)kvh * g.rot_stride(), D * D * sizeof(float), bar);
  }
  __syncthreads();   // the barrier is initialised before any thread waits on it
  const WsView ws = ws_view(a);
  const int c4 = lane % LPC, sub = lane / LPC;
  for (int hh = warp; hh < gq; hh += kWarps) {
    const float* base = ws.part + ((size_t)b * g.Hq + (size_t)kvh * gq + hh) * stride * (D + 4);
    float M = -INFINITY;
    for (int i = lane; i < nslot; i += 32) M = fmaxf(M, __ldcg(base + (size_t)i * (D + 4)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 pl = make_float4(0.f, 0.f, 0.f, 0.f), rr = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    for (int i0 = sub; i0 < nslot; i0 += 8 * SPW) {
      float2 ml[8];
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * SPW;
        if (i < nslot) {
          ml[u] = __ldcg(reinterpret_cast<const float2*>(base + (size_t)i * (D + 4)));
          v[u] = __ldcg(reinterpret_cast<const float4*>(base + (size_t)i * (D + 4) + 4) + c4);
        } else {
          ml[u] = make_float2(-INFINITY, 0.f);
          v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * SPW;
        const float w = ml[u].x == -INFINITY ? 0.f : ex2(ml[u].x - M);
        L = fmaf(w, ml[u].y, L);
        if (i < wc) {
          pl.x = fmaf(w, v[u].x, pl.x); pl.y = fmaf(w, v[u].y, pl.y);
          pl.z = fmaf(w, v[u].z, pl.z); pl.w = fmaf(w, v[u].w, pl.w);
        } else {
          rr.x = fmaf(w, v[u].x, rr.x); rr.y = fmaf(w, v[u].y, rr.y);
          rr.z = fmaf(w, v[u].z, rr.z); rr.w = fmaf(w, v[u].w, rr.w);
        }
      }
    }
    if constexpr (SPW == 2) {   // the two halves of the warp took alternate partials
      pl.x += __shfl_xor_sync(0xffffffffu, pl.x, 16); pl.y += __shfl_xor_sync(0xffffffffu, pl.y, 16);
      pl.z += __shfl_xor_sync(0xffffffffu, pl.z, 16); pl.w += __shfl_xor_sync(0xffffffffu, pl.w, 16);
      rr.x += __shfl_xor_sync(0xffffffffu, rr.x, 16); rr.y += __shfl_xor_sync(0xffffffffu, rr.y, 16);
      rr.z += __shfl_xor_sync(0xffffffffu, rr.z, 16); rr.w += __shfl_xor_sync(0xffffffffu, rr.w, 16);
      L += __shfl_xor_sync(0xffffffffu, L, 16);
    }
    if (sub == 0) {
      *reinterpret_cast<float4*>(rot + hh * D + 4 * c4) = rr;
      *reinterpret_cast<float4*>(plain + hh * D + 4 * c4) = pl;
    }
    if (lane == 0) Ls[hh] = L;
  }
  const bool ok = mbar_wait_bounded(bar, 0, a.status);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) (void)mbar_wait_bounded(bar, 0, nullptr);   // drain the copy before exiting
    return;
  }
  constexpr int M4 = (D / 4) / NPK;   // float4 per k part
  const int j = tid % D, kp = tid / D;
  const float4* Rrow = reinterpret_cast<const float4*>(Rs + j * D);
  float acc[8];
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) acc[hh] = 0.f;
#pragma unroll 4
  for (int mm = 0; mm < M4; ++mm) {
    const int k4 = kp * M4 + (mm + j) % M4;
    const float4 r = Rrow[k4];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh < gq) {
        const float4 x = reinterpret_cast<const float4*>(rot + hh * D)[k4];
        acc[hh] = fmaf(x.x, r.x, fmaf(x.y, r.y, fmaf(x.z, r.z, fmaf(x.w, r.w, acc[hh]))));
      }
    }
  }
  if constexpr (NPK > 1) {
    if (kp == 1)
#pragma unroll
      for (int hh = 0; hh < 8; ++hh)
        if (hh < gq) xr[hh * D + j] = acc[hh];
    __syncthreads();
  }
  if (kp == 0) {
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      if (hh < gq) {
        float t = acc[hh];
        if constexpr (NPK > 1) t += xr[hh * D + j];
        const float L = Ls[hh];
        const float o = (plain[hh * D + j] + t) * (L > 0.f ? 1.f / L : 0.f);
        const size_t oi = ((size_t)b * g.Hq + (size_t)kvh * gq + hh) * D + j;
        if (a.out_dtype == kDtypeBF16) {
          __nv_bfloat16 hb = __float2bfloat16_rn(o);
          static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
        } else {
          static_cast<float*>(a.out)[oi] = o;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ INT2 split
// Page block of one (page, kv head), as stored in the pool:
//   K codes [P][D/4] | K (scale, zero) [P][D/32] | V codes [P][D/4] | V (scale, zero) [P][D/32]
template <int D, int NT, int P>
struct Int2Layout {
  static constexpr int ROW = D / 4;
  static constexpr int SZ = D / 8;
  static constexpr int KSZ = P * ROW;
  static constexpr int VC = KSZ + P * SZ;
  static constexpr int VSZ = VC + P * ROW;
  static constexpr int BLOCK = VSZ + P * SZ;
  static constexpr int GROUPS = D / 32;
  static constexpr int KT = D / 16;             // QK k-tiles
  static constexpr int MT = D / 16;             // PV m-tiles
  static constexpr int WS = P == 64 ? 2 : 4;    // ring stages per warp (one page block each)
  static constexpr int RING = kWarps * WS * BLOCK;
  static constexpr int PIDS = RING + kWarps * WS * (8 + 4);                       // per-warp page ids [kWarps][32]
  static constexpr int QOFF = (PIDS + kWarps * 32 * 4 + 15) / 16 * 16;  // after mbarriers, page-valid flags, page ids
  static constexpr int SMEM = QOFF + (NT == 1 ? KT * 32 * 8 : 0);  // + the NT = 1 query fragments
  // one-launch decode: the CTA's own query side (fragments [NT][KT][32], 2^-e and Q_g per
  // head); the query side's scratch over the ring stages 1.. (empty until the query side is
  // done: the staggered fill requests them afterwards) when they are large enough, else after
  // the rest; at the end, in the CTA that merges, the merge's arrays from offset 0.
  static constexpr int QF = (SMEM + 15) / 16 * 16;
  static constexpr int QAUX = QF + NT * KT * 32 * 8;
  static constexpr int QR_BYTES = kQSideSmemFloats<D>() * 4;
  static constexpr bool QR_ALIAS = (WS - 1) * kWarps * BLOCK >= QR_BYTES;
  static constexpr int QR = QR_ALIAS ? kWarps * BLOCK : (QAUX + 8 * 8 * 4 + 15) / 16 * 16;
  static constexpr int FUSED_END = QR_ALIAS ? QAUX + 8 * 8 * 4 : QR + QR_BYTES;
  static constexpr int MERGE_END = kMergeSmemBytes<D>();
  static constexpr int SMEM_FUSED = FUSED_END > MERGE_END ? FUSED_END : MERGE_END;
};

// Speculative L2 prefetch before a one-launch decode's dependency wait (lane 0 of
// warp `warp`): an INT2 split CTA's warp prefetches its first page block, a window
// CTA's warp 0 (1) the chunk's K (V) rows.  Every index is checked against its
// buffer, so values the preceding grid has not finished writing give at worst a
// useless prefetch.
template <int P, int BLOCK>
__device__ __forceinline__ void prefetch_first_reads(const DecodeArgs& a, int b, int kvh, int warp) {
  const Geom& g = a.g;
  const int x = blockIdx.x;
  if (x < a.wl.win_chunks) {
    if (warp > 1) return;
    const int req = a.req_slot[b];
    const int t0 = x * kWinChunk;
    const int cnt = min(kWinChunk, g.window() - t0);
    if (req < 0 || req >= g.max_req || cnt <= 0) return;
    const size_t sbase = ((size_t)a.layer * g.max_req + req) * g.slab_req_elems();
    bulk_prefetch_l2(a.slab + sbase + ((size_t)kvh * 2 + warp) * g.window() * g.D + (size_t)t0 * g.D,
                     (uint32_t)(cnt * g.D * 2));
    return;
  }
  const int n = a.seq_lens[b];
  const int h_end = n - g.W;
  if (n < 0 || n > a.max_seq || h_end <= g.S) return;
  const int lp = (x - a.wl.win_chunks) * a.wl.pages_per_split + warp;
  if (lp > (h_end - 1) / P || lp >= a.bt_stride || lp >= g.max_pages_per_req) return;
  const int pid = a.block_table[(size_t)b * a.bt_stride + lp];
  if (pid < 0 || pid >= g.num_pages) return;
  bulk_prefetch_l2(a.pool + (size_t)a.layer * g.layer_pool_bytes() + ((size_t)pid * g.Hkv + kvh) * BLOCK, BLOCK);
}

// One INT2 split: pages [pg0, pg1) of one (request, kv head).  Warp w owns pages
// pg0 + w + 4i and streams them through its own ring of WS page blocks (bulk
// copies completing on per-stage mbarriers), so warps never wait on each other
// inside the loop.  A page is processed as P/16 blocks of 16 tokens.
//
// Operands (mma.sync m16n8k16, f32 accumulate).  Let k_K, k_V be the layer's
// operand exponents (scales and zeros times 2^k stay below 2^14 in f16), e_h the
// per-head query exponent written by q_rotate, and j = 6 the softmax-weight shift.
//   QK  A = K codes as f16 subnormals c * 2^(pos-24), one LOP3 per register
//       (exact, no offset term); B = q' * 2^(e_h) * 2^(10-pos) split into f16
//       hi/lo, so each product is c * q' * 2^(e_h - 14) exactly.  One accumulator
//       per 32-channel group; after its MMAs it is multiplied by the group's
//       scale s * 2^(k_K + 14) (float32 from the BF16 bits) and summed.  The zero
//       term sum_g z_g Q_g is one more MMA: A = the raw BF16 (scale, zero) word of
//       group tig in columns (2tig, 2tig+1), repeated in the upper k-half,
//       B = (0, Q_tig * 2^(e_h + k_K)) as three BF16 terms, the scale meeting a
//       zero row.
//   PV  A = V codes times their token's group scale (as for K, per token pair);
//       B = p * 2^j split into f16 hi/lo; the zero term sum_t p_t z_{t,g} is one
//       MMA with A rows = groups holding f16(z * 2^k_V).
//   Columns: <= 4 query heads: (head, hi|lo); 8 query heads: heads, with the hi
//   and lo planes as two MMAs into the same accumulator.
// Token order inside a 16-token block: MMA row / PV k-index r is token
// sigma(r) = r/2 + 8(r%2), which lets the PV weights of a lane come from two
// lanes' QK accumulators.
// Online softmax in the log2 domain with a lazy reference mm: it moves only
// when a block maximum exceeds mm + 8 + j, so weights 2^(s - mm) stay below
// 2^14 (f16) and rescaling is rare; the reference check is one warp vote.
// Returns false if a page copy timed out (the CTA then writes no partial).
// FUSED: the one-launch decode (the CTA forms its query side itself, window CTAs
// read q from the call's input; see q_side_cta and fused_merge).
template <int D, int NT, int P, bool FUSED>
__device__ __forceinline__ bool splitk_work(const DecodeArgs& a, uint8_t* smem) {
  using Lay = Int2Layout<D, NT, P>;
  constexpr int WS = Lay::WS;
  constexpr int GROUPS = Lay::GROUPS;
  constexpr bool G8 = NT == 2;
  constexpr int NH = G8 ? 2 : 1;  // query heads per lane

  const Geom& g = a.g;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int gq = g.gq();
  if (!a.pages_before_wait) {
    // The preceding grid is the caller's and may write anything this CTA reads
    // (lengths, block table, slots, pages).  Before waiting on it, lane 0 of each
    // warp brings the data it will most likely read first into L2, from the view
    // of those tables it has now: a stale view costs a useless prefetch, never a
    // wrong result (every read that counts comes after the wait).
    if (lane == 0) prefetch_first_reads<P, Int2Layout<D, NT, P>::BLOCK>(a, b, kvh, warp);
    pdl_wait();
  }
  const int n = a.seq_lens[b];
  if (!seq_len_ok(a, n)) {
    if (tid == 0 && blockIdx.x == 0) flag_error(a.status, kDevBadLen);
    pdl_launch_dependents();
    return true;
  }
  if ((int)blockIdx.x < a.wl.win_chunks) {
    const int req = a.req_slot[b];
    if (req < 0 || req >= g.max_req) {
      if (tid == 0 && blockIdx.x == 0) flag_error(a.status, kDevBadSlot);
      pdl_launch_dependents();
      return true;
    }
    pdl_wait();
    window_chunk<D, kThreads, FUSED>(a, b, kvh, blockIdx.x, smem, tid, [] { __syncthreads(); });
    pdl_launch_dependents();
    return true;
  }
  const int split = blockIdx.x - a.wl.win_chunks;
  const int h_end = n - g.W;
  if (h_end <= g.S) { pdl_launch_dependents(); return true; }
  const int n_hist_pages = (h_end - 1) / P + 1;
  const int pg0 = split * a.wl.pages_per_split;
  if (pg0 >= n_hist_pages) { pdl_launch_dependents(); return true; }
  const int pg1 = min(pg0 + a.wl.pages_per_split, n_hist_pages);
  const int n_mine = pg0 + warp < pg1 ? (pg1 - pg0 - warp + kWarps - 1) / kWarps : 0;

  const int* bt = a.block_table + (size_t)b * a.bt_stride;
  const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();
  // ring stage s of this warp (stage-major: every warp's stage 0, then every warp's stage 1, ...)
  auto stage_buf = [&](int s) { return smem + (s * kWarps + warp) * Lay::BLOCK; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::RING) + warp * WS;
  int* stage_ok = reinterpret_cast<int*>(smem + Lay::RING + kWarps * WS * 8) + warp * WS;

  // the page ids of this warp's first 32 pages, read once (lane i: page i), so that
  // refilling the ring needs no dependent global load
  int* pidtab = reinterpret_cast<int*>(smem + Lay::PIDS) + warp * 32;
  auto page_id = [&](int i) {
    const int lp = pg0 + warp + kWarps * i;
    return (lp < a.bt_stride && lp < g.max_pages_per_req) ? bt[lp] : -1;
  };
  if (lane < n_mine) pidtab[lane] = page_id(lane);
  if (lane == 0) {
    for (int s = 0; s < WS; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  const uint64_t stream_policy = l2_evict_first_policy();  // pages are read once per step
  auto issue = [&](int i) {  // lane 0: page i of this warp into stage i % WS
    const int s = i % WS;
    const int pid = i < 32 ? pidtab[i] : page_id(i);
    const bool okp = pid >= 0 && pid < g.num_pages;
    stage_ok[s] = okp ? 1 : 0;
    if (!okp) flag_error(a.status, kDevBadPage);
    mbar_arrive_expect_tx(&bars[s], okp ? (uint32_t)Lay::BLOCK : 0u);
    if (okp)
      bulk_g2s_hint(stage_buf(s), pool_l + ((size_t)pid * g.Hkv + kvh) * Lay::BLOCK, Lay::BLOCK, &bars[s],
                    stream_policy);
  };

  // The warp's first page is requested before the wait on the preceding grid, so
  // the page stream overlaps it; the rest of the ring is requested after that wait
  // and the query-side set-up (staggered fill: when every warp of the grid requests
  // its whole ring at once, each warp's first page lands only near the end of the
  // burst, while first pages requested first arrive first).  In a fused step the preceding
  // grid (the append) may still be writing the last history page: if that is the
  // first page, it is requested after the wait.  Behind a grid that is not this chain's
  // (pages_before_wait = 0) the CTA has waited already (see the top).
  auto is_tail = [&](int i) { return a.defer_tail_page && pg0 + warp + kWarps * i == n_hist_pages - 1; };
  int n_issued = 0;  // pages requested so far (lane 0)
  if (lane == 0 && n_mine > 0 && !is_tail(0)) {
    if (a.pages_before_wait) {
      issue(0);
      n_issued = 1;
    }
  }

  // ---------------- query side (written by q_rotate, or formed here): wait for the previous grid
  pdl_wait();
  if (lane == 0 && n_mine > 0 && n_issued == 0) {
    issue(0);
    n_issued = 1;
  }
  WsView ws = ws_view(a);
  uint2* qf_s = reinterpret_cast<uint2*>(smem + Lay::QF);     // one-launch decode: [NT][KT][32]
  float* qaux_s = reinterpret_cast<float*>(smem + Lay::QAUX);  // one-launch decode: [gq][8]
  if constexpr (FUSED) q_side_cta<D, NT>(a, kvh, b, reinterpret_cast<float*>(smem + Lay::QR), qf_s, qaux_s);
  // The query-side B fragments are the same for every warp of the CTA.  With up to
  // four query heads (NT = 1) they are staged once in shared memory (one LDS.64 per
  // MMA): the registers they free buy the 128-register kernel scheduling room.  With
  // eight heads (NT = 2) the kernel runs at three CTAs per SM with registers to
  // spare, and register operands avoid the extra loads.
  uint2* qsm = reinterpret_cast<uint2*>(smem + (FUSED ? Lay::QF : Lay::QOFF));   // [NT][KT][32 lanes]
  uint32_t qb[G8 ? NT : 1][G8 ? Lay::KT : 1][2];
  if constexpr (G8) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int kk = 0; kk < Lay::KT; ++kk) {
        const uint2 f = FUSED ? qf_s[(nt * Lay::KT + kk) * 32 + lane]
                              : ws.qfrag[((((size_t)b * g.Hkv + kvh) * NT + nt) * Lay::KT + kk) * 32 + lane];
        qb[nt][kk][0] = f.x;
        qb[nt][kk][1] = f.y;
      }
  } else if constexpr (!FUSED) {   // (the one-launch query side is in qsm already, absent heads zero)
    for (int i = tid; i < NT * Lay::KT * 32; i += kThreads) {
      const int nt = i / (Lay::KT * 32), rem = i % (Lay::KT * 32);
      const int kk = rem >> 5, ln = rem & 31;
      const bool col_ok = ((ln >> 2) >> 1) < gq;
      const uint2 f = ws.qfrag[((((size_t)b * g.Hkv + kvh) * NT + nt) * Lay::KT + kk) * 32 + ln];
      qsm[i] = col_ok ? f : make_uint2(0u, 0u);
    }
    __syncthreads();
  }
  const float* aux_base = FUSED ? qaux_s : ws.qaux + ((size_t)b * g.Hq + (size_t)kvh * gq) * 8;
  const float sm_log2 = kLog2e * rsqrtf((float)D);
  float F[NH];  // score = accumulator * F (log2 domain)
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const int hh = G8 ? 2 * tig + j : tig;
    F[j] = hh < gq ? aux_base[hh * 8] * ldexpf(sm_log2, -a.k_exp_K) : 0.f;
  }
  // zero-term B fragments: column gid, row 2tig + 1 = Q_tig * 2^(e_h + k_K) as three BF16
  // terms (hi + lo + lo2, 24 bits): part 0 carries hi in rows 0..7 (qz) and lo2 in rows
  // 8..15 (qz2), part 1 carries lo; the A rows 8..15 repeat the (s, z) words.  Two terms
  // (16 bits) leave errors of a few 1e-3 of the output's RMS at 32K tokens.
  uint32_t qz[NT], qz2[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = G8 ? gid : gid >> 1;
    const int part = G8 ? nt : gid & 1;
    float v = 0.f, v2 = 0.f;
    if (hh < gq && tig < GROUPS) {
      const float* aux = aux_base + hh * 8;
      const float qf = ldexpf(aux[1 + tig] / aux[0], a.k_exp_K);
      const float hi = __bfloat162float(__float2bfloat16_rn(qf));
      const float lo = __bfloat162float(__float2bfloat16_rn(qf - hi));
      v = part ? lo : hi;
      v2 = part ? 0.f : qf - hi - lo;
    }
    const __nv_bfloat16 vb = __float2bfloat16_rn(v), vb2 = __float2bfloat16_rn(v2);
    qz[nt] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&vb)) << 16;
    qz2[nt] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&vb2)) << 16;
  }

  // the rest of the ring, a query-side set-up later than the first pages of the grid
  if (lane == 0)
    for (; n_issued < WS && n_issued < n_mine; ++n_issued) issue(n_issued);

  float mm[NH], thr[NH], l_run[NH];
  float acc[Lay::MT][4];
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    mm[j] = -INFINITY;
    thr[j] = -INFINITY;
    l_run[j] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;

  const uint32_t magic = a.code_magic;
  const uint32_t k23 = static_cast<uint32_t>(a.k_exp_K + 14) << 23;   // K scales: s * 2^(k_K + 14)
  const uint32_t v23 = static_cast<uint32_t>(a.k_exp_V) << 23;
  // rows of this lane inside a 16-token block: QK rows gid, gid + 8 are tokens
  // ra = sigma(gid), rb = sigma(gid + 8); PV k-indices 2tig, 2tig+1, 2tig+8, 2tig+9
  // are tokens tig, tig + 8, tig + 4, tig + 12
  const int ra = (gid >> 1) + 8 * (gid & 1);
  const int rb = ra + 4;
  const int zq = min(tig, GROUPS - 1);   // QK zero-term group of this lane
  const int zv = gid & (GROUPS - 1);     // PV zero-term group row of this lane
  const int src0 = (2 * tig) * 4 + (gid >> 1), src1 = src0 + 4;
  const uint32_t psel = (gid & 1) ? 0x7632u : 0x5410u;
  // this lane's byte offsets inside a 16-token block of a stage buffer, relative to
  // the block's code rows (pc) or (scale, zero) rows (ps): K row ra (row rb is 4 rows
  // on), V token tig (tokens tig + 8, tig + 4, tig + 12 are 8, 4, 12 rows on)
  const int oK = ra * Lay::ROW + (D == 128 ? tig * 8 : tig * 4);
  const int oKs = Lay::KSZ + ra * Lay::SZ;
  const int oKz = oKs + 4 * zq;
  const int oV = Lay::VC + tig * Lay::ROW + (D == 128 ? gid * 4 : (gid >> 1) * 4);
  const int oVs = Lay::VSZ + tig * Lay::SZ;
  const int oVz = oVs + 4 * zv;

  // One 16-token block at slot0 of the stage buffer; FULL: every token is a
  // history token (no masking).
  // ---------------- QK scores of one 16-token block at slot0 of a stage buffer
  // (log2 domain, masked to -inf outside the history unless FULL)
  struct Scores {
    float a[NH], b[NH];  // rows ra, rb of the block, per query head of the lane
  };
  auto qk = [&](auto full_tag, const uint8_t* buf, int slot0, int tb) -> Scores {
    constexpr bool FULL = decltype(full_tag)::value;
    Scores sc;
    float* sa = sc.a;
    float* sb = sc.b;
    const uint8_t* pc = buf + slot0 * Lay::ROW;
    const uint8_t* ps = buf + slot0 * Lay::SZ;
    bool va = true, vb = true;
    if constexpr (!FULL) {
      va = tb + ra >= g.S && tb + ra < h_end;
      vb = tb + rb >= g.S && tb + rb < h_end;
    }
    uint32_t kwA[D / 64], kwB[D / 64];
    uint32_t szA[GROUPS], szB[GROUPS];
    if constexpr (D == 128) {
      const uint2 x = *reinterpret_cast<const uint2*>(pc + oK);
      const uint2 y = *reinterpret_cast<const uint2*>(pc + oK + 4 * Lay::ROW);
      kwA[0] = x.x; kwA[1] = x.y; kwB[0] = y.x; kwB[1] = y.y;
      const uint4 A4 = *reinterpret_cast<const uint4*>(ps + oKs);
      const uint4 B4 = *reinterpret_cast<const uint4*>(ps + oKs + 4 * Lay::SZ);
      szA[0] = A4.x; szA[1] = A4.y; szA[2] = A4.z; szA[3] = A4.w;
      szB[0] = B4.x; szB[1] = B4.y; szB[2] = B4.z; szB[3] = B4.w;
    } else {
      kwA[0] = *reinterpret_cast<const uint32_t*>(pc + oK);
      kwB[0] = *reinterpret_cast<const uint32_t*>(pc + oK + 4 * Lay::ROW);
      const uint2 A2 = *reinterpret_cast<const uint2*>(ps + oKs);
      const uint2 B2 = *reinterpret_cast<const uint2*>(ps + oKs + 4 * Lay::SZ);
      szA[0] = A2.x; szA[1] = A2.y;
      szB[0] = B2.x; szB[1] = B2.y;
    }
    uint32_t zA = *reinterpret_cast<const uint32_t*>(ps + oKz);
    uint32_t zB = *reinterpret_cast<const uint32_t*>(ps + oKz + 4 * Lay::SZ);
    // group scales s * 2^(k_K + 14), applied to each group's accumulator after its MMAs
    float SA[GROUPS], SB[GROUPS];
#pragma unroll
    for (int gi = 0; gi < GROUPS; ++gi) {
      SA[gi] = scale_times_pow2(szA[gi], k23);
      SB[gi] = scale_times_pow2(szB[gi], k23);
    }
    if constexpr (!FULL) {
      zA = va ? zA : 0u;
      zB = vb ? zB : 0u;
    }
    // per group: sum_c code_c * q'_c * 2^(e - 14) over its 32 channels (codes as exact
    // f16 subnormals); the zero term sum_g z_g Q_g * 2^(e + k) in its own accumulator
    float c[GROUPS][4];
    float cz[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int gi = 0; gi < GROUPS; ++gi) c[gi][0] = c[gi][1] = c[gi][2] = c[gi][3] = 0.f;
#pragma unroll
    for (int w = 0; w < D / 64; ++w) {
      const uint32_t a6 = kwA[w] >> 6, b6 = kwB[w] >> 6;
      uint32_t ua[8], ub[8];
#define OSCAR_K_SLOT(X)                        \
      ua[X] = subnormal_slot<X>(kwA[w], a6); \
      ub[X] = subnormal_slot<X>(kwB[w], b6);
      OSCAR_K_SLOT(0) OSCAR_K_SLOT(1) OSCAR_K_SLOT(2) OSCAR_K_SLOT(3)
      OSCAR_K_SLOT(4) OSCAR_K_SLOT(5) OSCAR_K_SLOT(6) OSCAR_K_SLOT(7)
#undef OSCAR_K_SLOT
#pragma unroll
      for (int hg = 0; hg < 2; ++hg) {
        const int gi = 2 * w + hg;
#pragma unroll
        for (int kt = 0; kt < 2; ++kt) {
          const int x = 4 * hg + 2 * kt;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
          if constexpr (G8) {
            mma_f16(c[gi], ua[x], ub[x], ua[x + 1], ub[x + 1], qb[nt][2 * gi + kt][0], qb[nt][2 * gi + kt][1]);
          } else {
            const uint2 qf = qsm[(nt * Lay::KT + 2 * gi + kt) * 32 + lane];
            mma_f16(c[gi], ua[x], ub[x], ua[x + 1], ub[x + 1], qf.x, qf.y);
          }
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_bf16(cz, zA, zB, zA, zB, qz[nt], qz2[nt]);
    if constexpr (G8) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float ta = cz[j], tb = cz[2 + j];
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi) {
          ta = fmaf(SA[gi], c[gi][j], ta);
          tb = fmaf(SB[gi], c[gi][2 + j], tb);
        }
        sa[j] = ta * F[j];
        sb[j] = tb * F[j];
      }
    } else {
      float ta = cz[0] + cz[1], tb = cz[2] + cz[3];
#pragma unroll
      for (int gi = 0; gi < GROUPS; ++gi) {
        ta = fmaf(SA[gi], c[gi][0] + c[gi][1], ta);
        tb = fmaf(SB[gi], c[gi][2] + c[gi][3], tb);
      }
      sa[0] = ta * F[0];
      sb[0] = tb * F[0];
    }
    if constexpr (!FULL) {
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        sa[j] = va ? sa[j] : -INFINITY;
        sb[j] = vb ? sb[j] : -INFINITY;
      }
    }
    return sc;
  };
  // ---------------- online softmax: the reference moves (and the accumulators are
  // rescaled) only when a lane's block maximum mloc exceeds the threshold
  auto update_ref = [&](float m0, float m1) {
    const float mloc[2] = {m0, m1};
    bool need = false;
#pragma unroll
    for (int j = 0; j < NH; ++j) need |= mloc[j] > thr[j];
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        float mb = mloc[j];
        mb = warp_max_xor(mb, 4);
        mb = warp_max_xor(mb, 8);
        mb = warp_max_xor(mb, 16);
        const float nm = mb > thr[j] ? mb - kWeightShift : mm[j];
        const float alpha = nm == mm[j] ? 1.f : ex2(mm[j] - nm);
        mm[j] = nm;
        thr[j] = nm + kWeightShift + kRescaleLog2;
        l_run[j] *= alpha;
        if constexpr (G8) {
#pragma unroll
          for (int mt = 0; mt < Lay::MT; ++mt) {
            acc[mt][j] *= alpha;
            acc[mt][2 + j] *= alpha;
          }
          zacc[j] *= alpha;
          zacc[2 + j] *= alpha;
        } else {
#pragma unroll
          for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][r] *= alpha;
#pragma unroll
          for (int r = 0; r < 4; ++r) zacc[r] *= alpha;
        }
      }
    }
  };
  // ---------------- weights 2^(s - mm) of one block's scores, their sum, and PV
  auto pv = [&](auto full_tag, const uint8_t* buf, int slot0, int tb, const Scores& sc) {
    constexpr bool FULL = decltype(full_tag)::value;
    const float* sa = sc.a;
    const float* sb = sc.b;
    const uint8_t* pc = buf + slot0 * Lay::ROW;
    const uint8_t* ps = buf + slot0 * Lay::SZ;
    float pa[NH], pb[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      pa[j] = ex2(sa[j] - mm[j]);
      pb[j] = ex2(sb[j] - mm[j]);
      l_run[j] += pa[j] + pb[j];
    }
    // ---------------- PV weights: f16 hi/lo of p, moved to the B layout
    uint32_t bw[NT][2];
    if constexpr (G8) {
      const uint32_t ha = pack_half2(pa[0], pa[1]), hb = pack_half2(pb[0], pb[1]);
      const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&ha));
      const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&hb));
      const uint32_t la = pack_half2(pa[0] - fa.x, pa[1] - fa.y), lb = pack_half2(pb[0] - fb.x, pb[1] - fb.y);
      bw[0][0] = prmt(__shfl_sync(0xffffffffu, ha, src0), __shfl_sync(0xffffffffu, ha, src1), psel);
      bw[0][1] = prmt(__shfl_sync(0xffffffffu, hb, src0), __shfl_sync(0xffffffffu, hb, src1), psel);
      bw[NT - 1][0] = prmt(__shfl_sync(0xffffffffu, la, src0), __shfl_sync(0xffffffffu, la, src1), psel);
      bw[NT - 1][1] = prmt(__shfl_sync(0xffffffffu, lb, src0), __shfl_sync(0xffffffffu, lb, src1), psel);
    } else {
      const uint32_t h = pack_half2(pa[0], pb[0]);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&h));
      const uint32_t lo = pack_half2(pa[0] - hf.x, pb[0] - hf.y);
      const uint32_t hla = prmt(h, lo, 0x5410), hlb = prmt(h, lo, 0x7632);
      bw[0][0] = prmt(__shfl_sync(0xffffffffu, hla, src0), __shfl_sync(0xffffffffu, hla, src1), psel);
      bw[0][1] = prmt(__shfl_sync(0xffffffffu, hlb, src0), __shfl_sync(0xffffffffu, hlb, src1), psel);
    }
    // ---------------- PV
    bool v0 = true, v1 = true, v2 = true, v3 = true;
    if constexpr (!FULL) {
      v0 = tb + tig >= g.S && tb + tig < h_end;
      v1 = tb + tig + 8 >= g.S && tb + tig + 8 < h_end;
      v2 = tb + tig + 4 >= g.S && tb + tig + 4 < h_end;
      v3 = tb + tig + 12 >= g.S && tb + tig + 12 < h_end;
    }
    uint32_t xw[D / 64], yw[D / 64];  // code words: tokens (r0 | r1) and (r2 | r3) per half-word
    if constexpr (D == 128) {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(pc + oV);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(pc + oV + 8 * Lay::ROW);
      const uint32_t w2 = *reinterpret_cast<const uint32_t*>(pc + oV + 4 * Lay::ROW);
      const uint32_t w3 = *reinterpret_cast<const uint32_t*>(pc + oV + 12 * Lay::ROW);
      xw[0] = prmt(w0, w1, 0x5410); xw[1] = prmt(w0, w1, 0x7632);
      yw[0] = prmt(w2, w3, 0x5410); yw[1] = prmt(w2, w3, 0x7632);
    } else {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(pc + oV);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(pc + oV + 8 * Lay::ROW);
      const uint32_t w2 = *reinterpret_cast<const uint32_t*>(pc + oV + 4 * Lay::ROW);
      const uint32_t w3 = *reinterpret_cast<const uint32_t*>(pc + oV + 12 * Lay::ROW);
      xw[0] = prmt(w0, w1, psel);
      yw[0] = prmt(w2, w3, psel);
    }
    uint32_t Sx[GROUPS], Sy[GROUPS];
    {
      uint32_t s0[GROUPS], s1[GROUPS], s2[GROUPS], s3[GROUPS];
      if constexpr (D == 128) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(ps + oVs);
        const uint4 q1 = *reinterpret_cast<const uint4*>(ps + oVs + 8 * Lay::SZ);
        const uint4 q2 = *reinterpret_cast<const uint4*>(ps + oVs + 4 * Lay::SZ);
        const uint4 q3 = *reinterpret_cast<const uint4*>(ps + oVs + 12 * Lay::SZ);
        s0[0] = q0.x; s0[1] = q0.y; s0[2] = q0.z; s0[3] = q0.w;
        s1[0] = q1.x; s1[1] = q1.y; s1[2] = q1.z; s1[3] = q1.w;
        s2[0] = q2.x; s2[1] = q2.y; s2[2] = q2.z; s2[3] = q2.w;
        s3[0] = q3.x; s3[1] = q3.y; s3[2] = q3.z; s3[3] = q3.w;
      } else {
        const uint2 q0 = *reinterpret_cast<const uint2*>(ps + oVs);
        const uint2 q1 = *reinterpret_cast<const uint2*>(ps + oVs + 8 * Lay::SZ);
        const uint2 q2 = *reinterpret_cast<const uint2*>(ps + oVs + 4 * Lay::SZ);
        const uint2 q3 = *reinterpret_cast<const uint2*>(ps + oVs + 12 * Lay::SZ);
        s0[0] = q0.x; s0[1] = q0.y; s1[0] = q1.x; s1[1] = q1.y;
        s2[0] = q2.x; s2[1] = q2.y; s3[0] = q3.x; s3[1] = q3.y;
      }
#pragma unroll
      for (int gi = 0; gi < GROUPS; ++gi) {
        float f0 = neg_scale_times_pow2(s0[gi], v23), f1 = neg_scale_times_pow2(s1[gi], v23);
        float f2 = neg_scale_times_pow2(s2[gi], v23), f3 = neg_scale_times_pow2(s3[gi], v23);
        if constexpr (!FULL) {
          f0 = v0 ? f0 : 0.f;
          f1 = v1 ? f1 : 0.f;
          f2 = v2 ? f2 : 0.f;
          f3 = v3 ? f3 : 0.f;
        }
        Sx[gi] = pack_half2(f0, f1);
        Sy[gi] = pack_half2(f2, f3);
      }
    }
    // ux[k] / uy[k]: half-word part k >> 3, slot k & 7 -> channel 64 (k >> 3) + 8 (k & 7) + gid, group k >> 2
    uint32_t ux[D / 8], uy[D / 8];
#pragma unroll
    for (int w = 0; w < D / 64; ++w) {
      const uint32_t x6 = xw[w] >> 6, y6 = yw[w] >> 6;
#define OSCAR_V_SLOT(X)                                                              \
      ux[8 * w + X] = scale_codes(magic_slot<X>(xw[w], x6, magic), Sx[(8 * w + X) >> 2]);    \
      uy[8 * w + X] = scale_codes(magic_slot<X>(yw[w], y6, magic), Sy[(8 * w + X) >> 2]);
      OSCAR_V_SLOT(0) OSCAR_V_SLOT(1) OSCAR_V_SLOT(2) OSCAR_V_SLOT(3)
      OSCAR_V_SLOT(4) OSCAR_V_SLOT(5) OSCAR_V_SLOT(6) OSCAR_V_SLOT(7)
#undef OSCAR_V_SLOT
    }
#pragma unroll
    for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_f16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bw[nt][0], bw[nt][1]);
    // zero term: rows = groups (row gid holds group zv), k = the lane's four tokens
    {
      float z0 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + oVz), v23);
      float z1 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + oVz + 8 * Lay::SZ), v23);
      float z2 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + oVz + 4 * Lay::SZ), v23);
      float z3 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + oVz + 12 * Lay::SZ), v23);
      if constexpr (!FULL) {
        z0 = v0 ? z0 : 0.f;
        z1 = v1 ? z1 : 0.f;
        z2 = v2 ? z2 : 0.f;
        z3 = v3 ? z3 : 0.f;
      }
      const uint32_t az0 = pack_half2(z0, z1), az2 = pack_half2(z2, z3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_f16(zacc, az0, 0u, az2, 0u, bw[nt][0], bw[nt][1]);
    }
  };
  // one block (masked pages)
  auto process = [&](auto full_tag, const uint8_t* buf, int slot0, int tb) {
    const Scores s0 = qk(full_tag, buf, slot0, tb);
    update_ref(fmaxf(s0.a[0], s0.b[0]), fmaxf(s0.a[NH - 1], s0.b[NH - 1]));
    pv(full_tag, buf, slot0, tb, s0);
  };
  // two blocks of a page wholly inside the history: both QK first (independent
  // work for the schedulers), one reference update for the 32 tokens, then PV
  auto process_pair = [&](const uint8_t* buf, int slot0, int tb) {
    const Scores s0 = qk(std::integral_constant<bool, true>{}, buf, slot0, tb);
    const Scores s1 = qk(std::integral_constant<bool, true>{}, buf, slot0 + 16, tb + 16);
    update_ref(fmaxf(fmaxf(s0.a[0], s0.b[0]), fmaxf(s1.a[0], s1.b[0])),
               fmaxf(fmaxf(s0.a[NH - 1], s0.b[NH - 1]), fmaxf(s1.a[NH - 1], s1.b[NH - 1])));
    pv(std::integral_constant<bool, true>{}, buf, slot0, tb, s0);
    pv(std::integral_constant<bool, true>{}, buf, slot0 + 16, tb + 16, s1);
  };
  // the four blocks of a 64-token page wholly inside the history, one reference update
  auto process_quad = [&](const uint8_t* buf, int tb) {
    const Scores s0 = qk(std::integral_constant<bool, true>{}, buf, 0, tb);
    const Scores s1 = qk(std::integral_constant<bool, true>{}, buf, 16, tb + 16);
    const Scores s2 = qk(std::integral_constant<bool, true>{}, buf, 32, tb + 32);
    const Scores s3 = qk(std::integral_constant<bool, true>{}, buf, 48, tb + 48);
    float m[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int jj = j < NH ? j : NH - 1;
      m[j] = fmaxf(fmaxf(fmaxf(s0.a[jj], s0.b[jj]), fmaxf(s1.a[jj], s1.b[jj])),
                   fmaxf(fmaxf(s2.a[jj], s2.b[jj]), fmaxf(s3.a[jj], s3.b[jj])));
    }
    update_ref(m[0], m[1]);
    pv(std::integral_constant<bool, true>{}, buf, 0, tb, s0);
    pv(std::integral_constant<bool, true>{}, buf, 16, tb + 16, s1);
    pv(std::integral_constant<bool, true>{}, buf, 32, tb + 32, s2);
    pv(std::integral_constant<bool, true>{}, buf, 48, tb + 48, s3);
  };

  bool aborted = false;
  int i_fail = 0;
  for (int i = 0; i < n_mine; ++i) {
    const int s = i % WS;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_sleep_bounded(&bars[s], (i / WS) & 1, a.status));
    if (!ok) {
      aborted = true;
      i_fail = i;
      break;
    }

    if (stage_ok[s]) {
      const uint8_t* buf = stage_buf(s);
      const int tp = (pg0 + warp + kWarps * i) * P;  // first token of the page
      if (tp >= g.S && tp + P <= h_end) {  // every token of the page is history: no checks
        if constexpr (P == 64) {
          process_quad(buf, tp);
        } else if constexpr (P == 32) {
          process_pair(buf, 0, tp);
        } else {
          process(std::integral_constant<bool, true>{}, buf, 0, tp);   // a 16-token page is one block
        }
      } else {
#pragma unroll 1
        for (int blk = 0; blk < P / 16; ++blk) {
          const int tb = tp + 16 * blk;
          if (tb + 16 > g.S && tb < h_end) process(std::integral_constant<bool, false>{}, buf, 16 * blk, tb);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + WS < n_mine) {
      fence_proxy_async_smem();
      issue(i + WS);
      n_issued = i + WS + 1;
    }
  }
  if (aborted && lane == 0) {
    // drain this warp's copies still in flight before the CTA exits, again bounded
    for (int i = i_fail; i < n_issued; ++i) (void)mbar_wait_bounded(&bars[i % WS], (i / WS) & 1, nullptr);
  }
  if constexpr (FUSED) {   // the merge may reuse the barriers' shared memory
    if (lane == 0)
      for (int st = 0; st < WS; ++st) mbar_inval(&bars[st]);
  }
  pdl_launch_dependents();
  if (__syncthreads_or(aborted)) return false;

  // ---------------- per-warp finalisation
  // zero-term sums of head j for group gi live in lane (gid = gi, tig)
  float zs[NH];
#pragma unroll
  for (int j = 0; j < NH; ++j) zs[j] = G8 ? zacc[j] : zacc[0] + zacc[1];
  float zg[NH][GROUPS];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
#pragma unroll
    for (int gi = 0; gi < GROUPS; ++gi) zg[j][gi] = __shfl_sync(0xffffffffu, zs[j], gi * 4 + tig);
  }
  // cross-warp merge through shared memory (every ring is idle now)
  float* wm = reinterpret_cast<float*>(smem);   // [4][8]
  float* wl = wm + 32;                          // [4][8]
  float* wacc = wl + 32;                        // [4][8][D]
  const float vscale = ldexpf(1.f, -a.k_exp_V);
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const int hh = G8 ? 2 * tig + j : tig;
    if (hh < gq) {
      if (gid == 0) {
        wm[warp * 8 + hh] = mm[j];
        wl[warp * 8 + hh] = l_run[j];
      }
#pragma unroll
      for (int mt = 0; mt < Lay::MT; ++mt) {
        const int ch_a = 16 * mt + gid, ch_b = ch_a + 8;
        const float va_ = G8 ? acc[mt][j] : acc[mt][0] + acc[mt][1];
        const float vb_ = G8 ? acc[mt][2 + j] : acc[mt][2] + acc[mt][3];
        // channel 16mt + gid (+ 8) sits in slot (2mt) mod 8 (+ 1) of its half-word:
        // code scale 2^(slot_pos - 10)
        const float za = zg[j][mt >> 1] * vscale;
        const float pa_ = static_cast<float>(1 << (10 - slot_pos((2 * mt) & 7)));   // folded after unrolling
        const float pb_ = static_cast<float>(1 << (10 - slot_pos((2 * mt + 1) & 7)));
        wacc[(warp * 8 + hh) * D + ch_a] = fmaf(va_, vscale * pa_, za);
        wacc[(warp * 8 + hh) * D + ch_b] = fmaf(vb_, vscale * pb_, za);
      }
    }
  }
  __syncthreads();
  // per head: the merged reference, the warps' weights and the merged sum
  float* wf = wacc + kWarps * 8 * D;   // [8][kWarps + 2]: f_0..f_3, M, L
  if (tid < gq) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * 8 + tid]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = wm[w * 8 + tid];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      wf[tid * (kWarps + 2) + w] = f;
      L = fmaf(f, wl[w * 8 + tid], L);
    }
    wf[tid * (kWarps + 2) + kWarps] = M;
    wf[tid * (kWarps + 2) + kWarps + 1] = L;
  }
  __syncthreads();
  const int stride = a.wl.win_chunks + a.wl.max_splits;
  for (int idx = tid; idx < gq * D; idx += kThreads) {
    const int hh = idx / D, ch = idx % D;
    const float* f = wf + hh * (kWarps + 2);
    float accv = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) accv = fmaf(f[w], wacc[(w * 8 + hh) * D + ch], accv);
    float* pp = ws.part + (((size_t)b * g.Hq + kvh * gq + hh) * stride + blockIdx.x) * (D + 4);
    pp[4 + ch] = accv;
    if (ch == 0) {
      pp[0] = f[kWarps];
      pp[1] = f[kWarps + 1];
    }
  }
  return true;
}

template <int D, int NT, int P, bool FUSED>
__global__ void __launch_bounds__(kThreads, 3) decode_splitk_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  (void)splitk_work<D, NT, P, FUSED>(a, smem);
  if constexpr (FUSED) {
    __shared__ int s_last;
    __shared__ __align__(8) uint64_t mbar;
    pdl_wait();          // (every path has waited already but the early exits) tickets follow the previous grid
    __threadfence();     // this thread's partial stores, device-wide, before the ticket
    __syncthreads();
    if (threadIdx.x == 0) {
      int* ctr = a.tickets + (size_t)blockIdx.z * a.g.Hkv + blockIdx.y;
      const bool last = atomicAdd(ctr, 1) == (int)gridDim.x - 1;
      if (last) {
        *ctr = 0;          // every CTA of the pair has its ticket: ready for the next launch
        __threadfence();   // the other CTAs' partials, seen through their tickets
      }
      s_last = last ? 1 : 0;
    }
    __syncthreads();
    if (s_last) fused_merge<D>(a, blockIdx.z, blockIdx.y, smem, &mbar);
  }
}

// ------------------------------------------------------------------ combine
// grid (Hq / hpc, B, D / jb), block kCombThreads.  One CTA merges the partials
// of hpc query heads of one request (window partials in the plain basis, INT2
// partials in the rotated basis) and produces output channels [j0, j0 + jb) of
// each: o_j = (plain_j + sum_k rot_k R_V[j][k]) / l.  Rows j0 .. j0 + jb of R_V
// and, when the plan says they fit, the heads' partials are staged in shared
// memory by bulk copies (R_V's before the wait on the split kernel).
//   1. warp per head: the reference M, the split weights 2^(m_i - M) and l;
//   2. every thread: merged rotated accumulators (all D channels) and the
//      window accumulators of its output channels;
//   3. thread per output channel (and head group, or k slice when the CTA has
//      fewer heads than threads per channel): float4 rows of R_V, each thread
//      starting at its own k offset so that a phase of 8 threads reads 8
//      different bank groups.
constexpr int kCombThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float csm[];
  __shared__ __align__(8) uint64_t bar;
  const Geom& g = a.g;
  const int hpc = a.wl.combine_hpc, jb = a.wl.combine_jb;
  const int b = blockIdx.y, h0 = blockIdx.x * hpc, j0 = blockIdx.z * jb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  WsView ws = ws_view(a);
  const int wc = a.wl.win_chunks;
  const int stride = wc + a.wl.max_splits;
  const size_t head_floats = (size_t)stride * (D + 4);
  float* Rs = csm;                             // [jb][D]: rows j0 .. j0 + jb of R_V
  float* rot = Rs + jb * D;                    // [hpc][D]
  float* plain = rot + hpc * D;                // [hpc][jb]
  float* red = plain + hpc * jb;               // [kCombThreads] k-slice partial sums
  float* lsum = red + kCombThreads;            // [16]
  float* parts = lsum + 16;                    // [hpc][stride][D + 4] when staged (16-byte aligned)
  float* wts = parts + (a.wl.combine_part_smem ? hpc * head_floats : 0);   // [hpc][stride]
  const float* gbase = ws.part + ((size_t)b * g.Hq + h0) * head_floats;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();  // the next kernel may launch and wait on this one
  const uint32_t r_bytes = (uint32_t)(jb * D * sizeof(float));
  const uint32_t p_bytes = a.wl.combine_part_smem ? (uint32_t)(hpc * head_floats * sizeof(float)) : 0u;
  // R_V does not depend on the previous kernel: start its copy before waiting on it
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, r_bytes + p_bytes);
    bulk_g2s(Rs, a.R_V + (size_t)(h0 / g.gq()) * g.rot_stride() + (size_t)j0 * D, r_bytes, &bar);
  }
  pdl_wait();
  if (tid == 0 && p_bytes) bulk_g2s(parts, gbase, p_bytes, &bar);
  const int n = a.seq_lens[b];
  const int nsp = seq_len_ok(a, n) ? min(splits_for(a, n), kMaxSplits) : 0;
  const int nslot = wc + nsp;
  const float* P = p_bytes ? parts : gbase;
  bool ok = true;
  if (p_bytes) ok = mbar_wait_bounded(&bar, 0, a.status);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) (void)mbar_wait_bounded(&bar, 0, nullptr);  // drain the copies before exiting
    return;
  }
  // 1. weights and l, warp per head
  for (int hi = warp; hi < hpc; hi += kCombThreads / 32) {
    const float* base = P + hi * head_floats;
    float M = -INFINITY;
    for (int i = lane; i < nslot; i += 32) M = fmaxf(M, base[(size_t)i * (D + 4)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i < nslot; i += 32) {
      const float mi = base[(size_t)i * (D + 4)];
      const float w = (mi == -INFINITY) ? 0.f : ex2(mi - M);
      wts[hi * stride + i] = w;
      L = fmaf(w, base[(size_t)i * (D + 4) + 1], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) lsum[hi] = L;
  }
  __syncthreads();
  // 2. merged accumulators: warp per head, lane per four channels; each slot is one
  //    float4 per lane and eight slots' loads are in flight at a time
  for (int hi = warp; hi < hpc; hi += kCombThreads / 32) {
    const float* base = P + hi * head_floats + 4;   // slot i, channel c: base[i * (D + 4) + c]
    const float* w = wts + hi * stride;
    for (int c4 = lane; c4 < D / 4; c4 += 32) {
      const int c = 4 * c4;
      float4 pl = make_float4(0.f, 0.f, 0.f, 0.f), r = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i < wc; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(base + (size_t)i * (D + 4) + c);
        const float wi = w[i];
        pl.x = fmaf(wi, v.x, pl.x); pl.y = fmaf(wi, v.y, pl.y); pl.z = fmaf(wi, v.z, pl.z); pl.w = fmaf(wi, v.w, pl.w);
      }
#pragma unroll 8
      for (int i = wc; i < nslot; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(base + (size_t)i * (D + 4) + c);
        const float wi = w[i];
        r.x = fmaf(wi, v.x, r.x); r.y = fmaf(wi, v.y, r.y); r.z = fmaf(wi, v.z, r.z); r.w = fmaf(wi, v.w, r.w);
      }
      *reinterpret_cast<float4*>(rot + hi * D + c) = r;
      const int cj = c - j0;
      if (cj >= 0 && cj < jb) *reinterpret_cast<float4*>(plain + hi * jb + cj) = pl;
    }
  }
  if (!p_bytes) ok = mbar_wait_bounded(&bar, 0, a.status);  // R_V rows
  if (!__syncthreads_and(ok)) {
    if (tid == 0) (void)mbar_wait_bounded(&bar, 0, nullptr);
    return;
  }
  // 3. R_V^T: thread (jl, r); heads split over head groups, or k over slices
  const int TJ = kCombThreads / jb;       // threads per output channel
  const int hg = TJ < hpc ? TJ : hpc;     // head groups
  const int KS = TJ / hg;                 // k slices per head group
  const int NHT = hpc / hg;               // heads per thread (at most 8)
  const int jl = tid % jb, r = tid / jb;
  const int grp = r / KS, slice = r % KS;
  const int m_per = (D / 4) / KS;
  const float4* Rrow = reinterpret_cast<const float4*>(Rs + jl * D);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int mm = 0; mm < m_per; ++mm) {
    const int k4 = slice * m_per + (mm + jl) % m_per;
    const float4 rr = Rrow[k4];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < NHT) {
        const float4 x = reinterpret_cast<const float4*>(rot + (grp + u * hg) * D)[k4];
        acc[u] = fmaf(x.x, rr.x, fmaf(x.y, rr.y, fmaf(x.z, rr.z, fmaf(x.w, rr.w, acc[u]))));
      }
    }
  }
  if (KS > 1) {  // one head per thread: sum the k slices
    red[tid] = acc[0];
    __syncthreads();
    if (slice == 0) {
      float s = 0.f;
      for (int sl = 0; sl < KS; ++sl) s += red[(grp * KS + sl) * jb + jl];
      acc[0] = s;
    }
  }
  if (slice == 0) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < NHT) {
        const int hi = grp + u * hg;
        const float L = lsum[hi];
        const float o = (plain[hi * jb + jl] + acc[u]) * (L > 0.f ? 1.f / L : 0.f);
        const size_t oi = ((size_t)b * g.Hq + h0 + hi) * D + j0 + jl;
        if (a.out_dtype == kDtypeBF16) {
          __nv_bfloat16 hb = __float2bfloat16_rn(o);
          static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
        } else {
          static_cast<float*>(a.out)[oi] = o;
        }
      }
    }
  }
}

// Small batches: one CTA per (query head, request), kHeadThreads threads.  R_V
// and the head's split partials are staged in shared memory by bulk copies
// (R_V's before the wait on the split kernel).  Warp 0 forms the split weights;
// NP = kHeadThreads / D threads per channel merge a share of the slots each;
// NP threads per output channel split R_V^T's k range (float4 rows, each thread
// starting at its own offset so that a phase of 8 threads reads 8 different
// bank groups).  The whole tail after the split kernel is a few short steps.
constexpr int kHeadThreads = 256;

template <int D>
__global__ void __launch_bounds__(kHeadThreads) decode_combine_head_kernel(DecodeArgs a) {
  constexpr int NP = kHeadThreads / D;
  extern __shared__ __align__(16) float csm[];
  float* Rs = csm;                 // [D][D]
  float* parts = Rs + D * D;       // [stride][D + 4] when staged
  __shared__ __align__(16) float rot[D];
  __shared__ float plain[D];
  __shared__ float share[NP][D];   // per-part sums (merge, then R_V^T)
  __shared__ float wts[kMaxSplits + kMaxWinChunks];
  __shared__ float s_l;
  __shared__ __align__(8) uint64_t bar;
  const Geom& g = a.g;
  const int b = blockIdx.y, h = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  WsView ws = ws_view(a);
  const int wc = a.wl.win_chunks;
  const int stride = wc + a.wl.max_splits;
  const size_t head_bytes = (size_t)stride * (D + 4) * sizeof(float);
  const float* gbase = ws.part + ((size_t)b * g.Hq + h) * stride * (D + 4);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();  // the next kernel may launch and wait on this one
  // R_V does not depend on the previous kernel: start its copy before waiting on it
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, D * D * sizeof(float) + (a.wl.combine_part_smem ? head_bytes : 0));
    bulk_g2s(Rs, a.R_V + (size_t)(h / g.gq()) * g.rot_stride(), D * D * sizeof(float), &bar);
  }
  pdl_wait();
  if (tid == 0 && a.wl.combine_part_smem) bulk_g2s(parts, gbase, (uint32_t)head_bytes, &bar);
  const int n = a.seq_lens[b];
  const int nsp = seq_len_ok(a, n) ? min(splits_for(a, n), kMaxSplits) : 0;
  const int nslot = wc + nsp;
  if (!mbar_wait_bounded(&bar, 0, a.status)) {
    (void)mbar_wait_bounded(&bar, 0, nullptr);
    return;
  }
  const float* base = a.wl.combine_part_smem ? parts : gbase;
  // 1. split weights and l (warp 0)
  if (warp == 0) {
    float M = -INFINITY;
    for (int i = lane; i < nslot; i += 32) M = fmaxf(M, base[(size_t)i * (D + 4)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i < nslot; i += 32) {
      const float mi = base[(size_t)i * (D + 4)];
      const float w = (mi == -INFINITY) ? 0.f : ex2(mi - M);
      wts[i] = w;
      L = fmaf(w, base[(size_t)i * (D + 4) + 1], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) s_l = L;
  }
  __syncthreads();
  // 2. merge: channel c, part p takes slots [lo, hi) of the INT2 splits; part 0 the window
  {
    const int c = tid % D, p = tid / D;
    const int nint = nslot - wc;
    const int lo = wc + nint * p / NP, hi = wc + nint * (p + 1) / NP;
    float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
    int i = lo;
    for (; i + 3 < hi; i += 4) {
      r0 = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + c], r0);
      r1 = fmaf(wts[i + 1], base[(size_t)(i + 1) * (D + 4) + 4 + c], r1);
      r2 = fmaf(wts[i + 2], base[(size_t)(i + 2) * (D + 4) + 4 + c], r2);
      r3 = fmaf(wts[i + 3], base[(size_t)(i + 3) * (D + 4) + 4 + c], r3);
    }
    for (; i < hi; ++i) r0 = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + c], r0);
    share[p][c] = (r0 + r1) + (r2 + r3);
    if (p == 0) {
      float q0 = 0.f, q1 = 0.f;
      int k = 0;
      for (; k + 1 < wc; k += 2) {
        q0 = fmaf(wts[k], base[(size_t)k * (D + 4) + 4 + c], q0);
        q1 = fmaf(wts[k + 1], base[(size_t)(k + 1) * (D + 4) + 4 + c], q1);
      }
      if (k < wc) q0 = fmaf(wts[k], base[(size_t)k * (D + 4) + 4 + c], q0);
      plain[c] = q0 + q1;
    }
  }
  __syncthreads();
  if (tid < D) {
    float r = 0.f;
#pragma unroll
    for (int p = 0; p < NP; ++p) r += share[p][tid];
    rot[tid] = r;
  }
  __syncthreads();
  // 3. (rot R_V^T)_j = sum_k rot_k R_V[j][k]: output j, k part kp
  {
    const int j = tid % D, kp = tid / D;
    constexpr int M4 = (D / 4) / NP;   // float4 per part
    const float4* Rrow = reinterpret_cast<const float4*>(Rs + j * D);
    const float4* r4 = reinterpret_cast<const float4*>(rot);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 4
    for (int mm = 0; mm < M4; mm += 2) {
      const int k4a = kp * M4 + (mm + j) % M4, k4b = kp * M4 + (mm + 1 + j) % M4;
      const float4 ra = Rrow[k4a], xa = r4[k4a], rb = Rrow[k4b], xb = r4[k4b];
      acc0 = fmaf(xa.x, ra.x, fmaf(xa.y, ra.y, fmaf(xa.z, ra.z, fmaf(xa.w, ra.w, acc0))));
      acc1 = fmaf(xb.x, rb.x, fmaf(xb.y, rb.y, fmaf(xb.z, rb.z, fmaf(xb.w, rb.w, acc1))));
    }
    share[kp][j] = acc0 + acc1;
  }
  __syncthreads();
  if (tid < D) {
    float o = plain[tid];
#pragma unroll
    for (int p = 0; p < NP; ++p) o += share[p][tid];
    o *= s_l > 0.f ? 1.f / s_l : 0.f;
    const size_t oi = ((size_t)b * g.Hq + h) * D + tid;
    if (a.out_dtype == kDtypeBF16) {
      __nv_bfloat16 hb = __float2bfloat16_rn(o);
      static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
    } else {
      static_cast<float*>(a.out)[oi] = o;
    }
  }
}

template <int D, int NT, int P, bool FUSED>
int launch_splitk_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  using Lay = Int2Layout<D, NT, P>;
  size_t smem = FUSED ? Lay::SMEM_FUSED : Lay::SMEM;
  const size_t win_smem = 2 * kWinChunk * D * sizeof(uint16_t) + 8 * D * sizeof(float);
  const size_t merge_smem = (64 + kWarps * 8 * D + 8 * (kWarps + 2)) * sizeof(float);
  if (win_smem > smem) smem = win_smem;
  if (merge_smem > smem) smem = merge_smem;
  smem = (smem + 127) & ~size_t(127);
  // three CTAs per SM (the plan sizes one wave as 3 x 152 CTAs).  The one-launch form needs the
  // largest shared-memory carveout for that; the three-kernel form keeps the default, which
  // its neighbours in the chain use too (an SM holds CTAs of one carveout at a time, so a
  // different one would keep the programmatic overlap from happening)
  static_assert(3 * (Lay::SMEM_FUSED + 128 + 1024) <= 228 * 1024, "three CTAs per SM");
  auto kern = decode_splitk_kernel<D, NT, P, FUSED>;
  cudaError_t e = ensure_smem_limit(kern, smem, FUSED);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.wl.win_chunks + a.wl.max_splits, a.g.Hkv, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  return (int)e;
}

template <int D, int NT, bool FUSED>
int launch_splitk_f(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  switch (a.g.P) {
    case 16: return launch_splitk_t<D, NT, 16, FUSED>(a, s, pdl);
    case 32: return launch_splitk_t<D, NT, 32, FUSED>(a, s, pdl);
    default: return launch_splitk_t<D, NT, 64, FUSED>(a, s, pdl);
  }
}

template <int D, int NT>
int launch_splitk_p(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  return a.wl.fused ? launch_splitk_f<D, NT, true>(a, s, pdl) : launch_splitk_f<D, NT, false>(a, s, pdl);
}

template <int D>
int launch_q_rotate_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.g.Hkv * (D / 32), a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return (int)cudaLaunchKernelEx(&cfg, q_rotate_kernel<D>, a);
}

}  // namespace

int static_decode_scratch(void** out, size_t* capacity) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // with this device current
    if (e != cudaSuccess) return (int)e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  *capacity = kStaticScratchBytes;
  return 0;
}

int launch_q_rotate(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return a.g.D == 128 ? launch_q_rotate_t<128>(a, s, pdl) : launch_q_rotate_t<64>(a, s, pdl);
}

int launch_decode_splitk(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nt = a.wl.nt;
  if (a.g.D == 128) return nt == 2 ? launch_splitk_p<128, 2>(a, s, pdl) : launch_splitk_p<128, 1>(a, s, pdl);
  return nt == 2 ? launch_splitk_p<64, 2>(a, s, pdl) : launch_splitk_p<64, 1>(a, s, pdl);
}


int launch_decode_combine(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  const bool per_head = a.wl.combine_head != 0;
  cfg.gridDim = per_head ? dim3(a.g.Hq, a.batch) : dim3(a.g.Hq / a.wl.combine_hpc, a.batch, a.g.D / a.wl.combine_jb);
  cfg.blockDim = dim3(per_head ? kHeadThreads : kCombThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.dynamicSmemBytes = a.wl.combine_smem;
  auto go = [&](auto kern) -> int {
    cudaError_t e = ensure_smem_limit(kern, a.wl.combine_smem);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, kern, a);
  };
  if (a.g.D == 128) return per_head ? go(decode_combine_head_kernel<128>) : go(decode_combine_kernel<128>);
  return per_head ? go(decode_combine_head_kernel<64>) : go(decode_combine_kernel<64>);
}

}  // namespace oscar
