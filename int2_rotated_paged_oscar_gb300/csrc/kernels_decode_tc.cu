// INT2 split-K decode with the query-key product on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- the serving
// kernel unpacks and dequantises the INT2 history, scores it in the rotated
// basis (the query is rotated once) and accumulates values in the rotated basis
// (R_V^T is applied once, in the combine), with no extra memory traffic; arXiv
// abstract -- fused decode kernel, batch-1 decode faster than BF16 by cutting KV
// memory traffic.
//
// One CTA = one INT2 split (pages [pg0, pg1) of one (request, kv head)), and, when
// blockIdx.x < win_chunks, also BF16 window chunk blockIdx.x.  The split's pages
// stream through a ring of 128-token tiles in shared memory (one non-multicast
// bulk copy per page block, completing on the tile's mbarrier).  Roles:
//   token warps 0-3   thread t owns token t of a tile (TMEM lane t).  It unpacks
//                     the token's K codes into TMEM as the A operand of the QK
//                     product (f16 subnormals c * 2^(pos-24): one LOP3 per code
//                     pair, exact), then, once the product is in TMEM, turns the
//                     token's per-(group, head) dot products into scores with the
//                     group scales and zeros, runs the online softmax (a CTA-wide
//                     lazy reference), and writes the token's weights (f16 hi/lo)
//                     into the B operand of the value product.
//   value warps 4-11  warp w owns 16-token block w - 4 of every tile: value codes
//                     times their BF16 scales (LOP3 + HFMA2 per pair) against the
//                     staged weights on mma.sync m16n8k16, float32 accumulators in
//                     registers; warps 4-7 first score the BF16 window chunk.
//   control warp 12   one thread: page-table reads, bulk copies, and the QK
//                     tcgen05.mma issue (A from TMEM, B = the query operand in
//                     shared memory, D = scores in TMEM), one commit per tile.
// QK product, per tile: S[t][n] = sum_k A[t][k] B[k][n], M = 128 tokens, K = D
// channels in 16-channel steps, N = 16 columns per window.  B is block-diagonal
// over the 32-channel quantisation groups: column n = (group, head, hi|lo) holds
// q' * 2^(e_h + 10 - pos) (f16 hi or lo) on its group's channels and 0 elsewhere,
// so each column is one group's code dot product and the BF16 group scale is
// applied afterwards in float32 by the token thread.
// All waits are bounded by %globaltimer; a timeout sets OSCAR_DEV_TIMEOUT, the
// CTA drains its copies and MMAs, frees its tensor memory and writes no partial.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

#include "tc_common.cuh"
#include "q_rotate.cuh"
#include "decode_window.cuh"

constexpr int kTile = 128;                       // history tokens per tile
constexpr int kTokWarps = 4;                     // one TMEM lane quarter each
constexpr int kPvWarps = kTile / 16;             // one 16-token block of a tile each
constexpr int kCtrlWarp = kTokWarps + kPvWarps;  // 12
constexpr int kTcThreads = 32 * (kCtrlWarp + 1); // 416
constexpr int kMaxStages = 16;
constexpr int kMaxSplitPages = 256;              // page-id table of a split (the host plan keeps to it)
constexpr int kBarTok = 1, kBarWin = 2, kBarJoin = 3;  // named barriers (0 is __syncthreads)

// ------------------------------------------------------------------ extra PTX wrappers
// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (valid after tmem_wait_ld).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A is read from tensor memory (lane = row, each
// 32-bit column a pair of consecutive K elements), B from its descriptor.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void bar_sync_named(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over nthreads threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ geometry
template <int D, int GQ>
struct TcCfg {
  static constexpr int NT = GQ == 8 ? 2 : 1;          // weight planes of the value product
  static constexpr int GROUPS = D / 32;
  static constexpr int KSTEPS = D / 16;
  static constexpr int MT = D / 16;
  static constexpr int ROW = D / 4, SZ = D / 8;      // code row / (scale, zero) row bytes per token
  static constexpr int STAGE = kTile * (3 * D / 4);  // one tile of page blocks (any page size)
  // score columns: (group, head, hi|lo); CG per group, GPW groups per 16-column window
  static constexpr int CG = 2 * GQ;
  static constexpr int GPW = CG >= 16 ? 1 : 16 / CG;
  static constexpr int NWIN = (GROUPS + GPW - 1) / GPW;
  static constexpr int SCOLS = 16 * NWIN;
  static constexpr int ACOLS = D / 2;                // A operand columns of one tile (f16 pairs)
  static constexpr int TM_A = 0, TM_S = 2 * ACOLS;   // TMEM: A[2] then S[2]
  static constexpr int TM_USED = 2 * ACOLS + 2 * SCOLS;
  static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128 : 256;
  // shared memory (offsets from a 1024-aligned base)
  static constexpr int BQ = 0;                                     // B of the QK product: SCOLS rows x D, sw128
  static constexpr int W = BQ + SCOLS * D * 2;                     // weights [2][kPvWarps][NT][32] uint2
  static constexpr int WIN = W + 2 * kPvWarps * NT * 32 * 8;       // window chunk staging
  static constexpr int MISC = WIN + 2 * kWinChunk * D * 2 + 8 * D * 4;
  // misc: alpha[2][8] f32, flag[2] i32, red[4][8] f32, mm[8] f32, lred[4][8] f32, pmask[16] u32,
  //       pid[kMaxSplitPages] i32, tmem slot, abort, Qs[GROUPS][8] f32
  static constexpr int M_ALPHA = MISC, M_FLAG = M_ALPHA + 64, M_RED = M_FLAG + 16, M_MM = M_RED + 128,
                       M_LRED = M_MM + 32, M_PMASK = M_LRED + 128, M_PID = M_PMASK + 4 * kMaxStages,
                       M_TMEM = M_PID + 4 * kMaxSplitPages, M_ABORT = M_TMEM + 4,
                       M_QS = (M_ABORT + 4 + 15) / 16 * 16;   // Qs [GROUPS][8] f32
  static constexpr int BAR = M_QS + GROUPS * 8 * 4;
  // barriers: full[16], empty[16], a_full[2], qk_done[2], s_empty[2], w_full[2], w_empty[2]
  static constexpr int RING = (BAR + 8 * (2 * kMaxStages + 10) + 127) / 128 * 128;
  static size_t smem_bytes(int stages) { return 1024 + RING + (size_t)stages * STAGE; }
};

// ------------------------------------------------------------------ value product of one 16-token block
// Per-lane constants of the value product (offsets inside a page block).
struct PvLane {
  int oV, oVs, oVz;
  uint32_t psel;
};

// acc += V^T(codes * scales) . weights over the 16 tokens at slot0 of the page block
// buf (absolute history position tb of its first token); zacc += the zero-term.
// wf: the block's weights, [NT][32 lanes] uint2 in the B-fragment layout.
// FULL: every token of the block is history (no masking).
template <int D, int GQ, bool FULL>
__device__ __forceinline__ void pv_block(const PvLane& L, const uint8_t* buf, int slot0, int tb, const uint2* wf,
                                         float (&acc)[D / 16][4], float (&zacc)[4], int S, int h_end, uint32_t magic,
                                         uint32_t v23, int lane) {
  using C = TcCfg<D, GQ>;
  constexpr int NT = C::NT, GROUPS = C::GROUPS, ROW = C::ROW, SZ = C::SZ;
  const int tig = lane & 3;
  const uint8_t* pc = buf + slot0 * ROW;
  const uint8_t* ps = buf + slot0 * SZ;
  uint32_t bw[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint2 f = wf[nt * 32 + lane];
    bw[nt][0] = f.x;
    bw[nt][1] = f.y;
  }
  bool v0 = true, v1 = true, v2 = true, v3 = true;
  if constexpr (!FULL) {
    v0 = tb + tig >= S && tb + tig < h_end;
    v1 = tb + tig + 8 >= S && tb + tig + 8 < h_end;
    v2 = tb + tig + 4 >= S && tb + tig + 4 < h_end;
    v3 = tb + tig + 12 >= S && tb + tig + 12 < h_end;
  }
  uint32_t xw[D / 64], yw[D / 64];  // code words: tokens (r0 | r1) and (r2 | r3) per half-word
  {
    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(pc + L.oV);
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(pc + L.oV + 8 * ROW);
    const uint32_t w2 = *reinterpret_cast<const uint32_t*>(pc + L.oV + 4 * ROW);
    const uint32_t w3 = *reinterpret_cast<const uint32_t*>(pc + L.oV + 12 * ROW);
    if constexpr (D == 128) {
      xw[0] = prmt(w0, w1, 0x5410); xw[1] = prmt(w0, w1, 0x7632);
      yw[0] = prmt(w2, w3, 0x5410); yw[1] = prmt(w2, w3, 0x7632);
    } else {
      xw[0] = prmt(w0, w1, L.psel);
      yw[0] = prmt(w2, w3, L.psel);
    }
  }
  uint32_t Sx[GROUPS], Sy[GROUPS];
  {
    uint32_t s0[GROUPS], s1[GROUPS], s2[GROUPS], s3[GROUPS];
    if constexpr (D == 128) {
      const uint4 q0 = *reinterpret_cast<const uint4*>(ps + L.oVs);
      const uint4 q1 = *reinterpret_cast<const uint4*>(ps + L.oVs + 8 * SZ);
      const uint4 q2 = *reinterpret_cast<const uint4*>(ps + L.oVs + 4 * SZ);
      const uint4 q3 = *reinterpret_cast<const uint4*>(ps + L.oVs + 12 * SZ);
      s0[0] = q0.x; s0[1] = q0.y; s0[2] = q0.z; s0[3] = q0.w;
      s1[0] = q1.x; s1[1] = q1.y; s1[2] = q1.z; s1[3] = q1.w;
      s2[0] = q2.x; s2[1] = q2.y; s2[2] = q2.z; s2[3] = q2.w;
      s3[0] = q3.x; s3[1] = q3.y; s3[2] = q3.z; s3[3] = q3.w;
    } else {
      const uint2 q0 = *reinterpret_cast<const uint2*>(ps + L.oVs);
      const uint2 q1 = *reinterpret_cast<const uint2*>(ps + L.oVs + 8 * SZ);
      const uint2 q2 = *reinterpret_cast<const uint2*>(ps + L.oVs + 4 * SZ);
      const uint2 q3 = *reinterpret_cast<const uint2*>(ps + L.oVs + 12 * SZ);
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
#define OSCAR_V_SLOT(X)                                                                   \
    ux[8 * w + X] = scale_codes(magic_slot<X>(xw[w], x6, magic), Sx[(8 * w + X) >> 2]); \
    uy[8 * w + X] = scale_codes(magic_slot<X>(yw[w], y6, magic), Sy[(8 * w + X) >> 2]);
    OSCAR_V_SLOT(0) OSCAR_V_SLOT(1) OSCAR_V_SLOT(2) OSCAR_V_SLOT(3)
    OSCAR_V_SLOT(4) OSCAR_V_SLOT(5) OSCAR_V_SLOT(6) OSCAR_V_SLOT(7)
#undef OSCAR_V_SLOT
  }
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      mma_f16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bw[nt][0], bw[nt][1]);
  // zero term: rows = groups (row gid holds group gid mod GROUPS), k = the lane's four tokens
  {
    float z0 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + L.oVz), v23);
    float z1 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + L.oVz + 8 * SZ), v23);
    float z2 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + L.oVz + 4 * SZ), v23);
    float z3 = zero_times_pow2(*reinterpret_cast<const uint32_t*>(ps + L.oVz + 12 * SZ), v23);
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
}

// ------------------------------------------------------------------ the kernel
template <int D, int GQ>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(DecodeArgs a) {
  using C = TcCfg<D, GQ>;
  constexpr int NT = C::NT, GROUPS = C::GROUPS, KSTEPS = C::KSTEPS, MT = C::MT;
  constexpr int ROW = C::ROW, SZ = C::SZ, STAGE = C::STAGE;
  constexpr int CG = C::CG, GPW = C::GPW, NWIN = C::NWIN, SCOLS = C::SCOLS;
  constexpr bool G8 = GQ == 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const Geom& g = a.g;
  const int b = blockIdx.z, kvh = blockIdx.y, x = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.seq_lens[b];
  if (!seq_len_ok(a, n)) {
    if (tid == 0 && x == 0 && kvh == 0) flag_error(a.status, kDevBadLen);
    pdl_launch_dependents();
    return;
  }
  bool do_win = x < a.wl.win_chunks;
  if (do_win) {
    const int req = a.req_slot[b];
    if (req < 0 || req >= g.max_req) {
      if (tid == 0 && x == 0) flag_error(a.status, kDevBadSlot);
      do_win = false;
    }
  }
  const int nsp = min(splits_for(a, n), kMaxSplits);
  const bool do_int2 = x < nsp;
  if (!do_int2) {
    // a window chunk only: four warps, the rest leave
    if (do_win && tid < 128) {
      pdl_wait();
      window_chunk<D, 128>(a, b, kvh, x, smem + C::WIN, tid, [] { bar_sync_named(kBarWin, 128); });
    }
    pdl_launch_dependents();
    return;
  }

  // ---------------- split geometry
  const int P = g.P;
  const int lgP = P == 64 ? 6 : (P == 32 ? 5 : 4);
  const int PPT = kTile >> lgP;                    // pages per tile
  const int BLOCK = P * (3 * D / 4);               // one (page, kv head) block
  const int KSZ = P * ROW, VC = KSZ + P * SZ, VSZ = VC + P * ROW;
  const int S = g.S;
  const int h_end = n - g.W;
  const int n_hist_pages = (h_end - 1) / P + 1;
  const int pg0 = x * a.wl.pages_per_split;
  const int pg1 = min(pg0 + a.wl.pages_per_split, n_hist_pages);
  const int npages = pg1 - pg0;
  const int ntiles = (npages + PPT - 1) / PPT;
  const int NS = a.wl.tc_stages;

  uint8_t* bq = smem + C::BQ;
  uint2* wbuf = reinterpret_cast<uint2*>(smem + C::W);
  float* alpha_s = reinterpret_cast<float*>(smem + C::M_ALPHA);
  int* flag_s = reinterpret_cast<int*>(smem + C::M_FLAG);
  float* red_s = reinterpret_cast<float*>(smem + C::M_RED);
  float* mm_s = reinterpret_cast<float*>(smem + C::M_MM);
  float* lred_s = reinterpret_cast<float*>(smem + C::M_LRED);
  uint32_t* pmask_s = reinterpret_cast<uint32_t*>(smem + C::M_PMASK);
  int* pid_s = reinterpret_cast<int*>(smem + C::M_PID);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::M_TMEM);
  volatile int* abort_s = reinterpret_cast<volatile int*>(smem + C::M_ABORT);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* a_full = bars + 2 * kMaxStages;
  uint64_t* qk_done = a_full + 2;
  uint64_t* s_empty = a_full + 4;
  uint64_t* w_full = a_full + 6;
  uint64_t* w_empty = a_full + 8;
  uint8_t* ring = smem + C::RING;

  // ---------------- set-up: barriers, tensor memory, zeroed weight buffers
  for (int i = tid; i < 2 * kPvWarps * NT * 32; i += kTcThreads) wbuf[i] = make_uint2(0u, 0u);
  if (warp == kCtrlWarp) {
    if (lane == 0) {
      for (int s = 0; s < kMaxStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], kPvWarps);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&a_full[i], kTokWarps);
        mbar_init(&qk_done[i], 1);
        mbar_init(&s_empty[i], kTokWarps);
        mbar_init(&w_full[i], kTokWarps);
        mbar_init(&w_empty[i], kPvWarps);
      }
      *abort_s = 0;
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(tmem_slot, C::TM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float sm_log2 = kLog2e * rsqrtf((float)D);
  WsView ws = ws_view(a);

  if (warp == kCtrlWarp) {
    // =============================== control: page ids, bulk copies, QK issue
    const int* bt = a.block_table + (size_t)b * a.bt_stride;
    for (int i = lane; i < npages; i += 32) {
      const int lp = pg0 + i;
      const int pid = (lp < a.bt_stride && lp < g.max_pages_per_req) ? bt[lp] : -1;
      const bool okp = pid >= 0 && pid < g.num_pages;
      if (!okp) flag_error(a.status, kDevBadPage);
      pid_s[i] = okp ? pid : -1;
    }
    __syncwarp();
    if (lane == 0) {
      const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();
      const uint64_t policy = l2_evict_first_policy();  // pages are read once per step
      const int tail = a.defer_tail_page ? n_hist_pages - 1 : -1;
      int deferred_tile = -1, deferred_k = 0;
      auto arm = [&](int j, bool defer) {  // tile j into stage j % NS
        const int s = j % NS;
        uint32_t mask = 0;
        for (int k = 0; k < PPT; ++k) {
          const int i = j * PPT + k;
          if (i < npages && pid_s[i] >= 0) mask |= 1u << k;
        }
        pmask_s[s] = mask;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(__popc(mask) * BLOCK));
        for (int k = 0; k < PPT; ++k) {
          if (!((mask >> k) & 1)) continue;
          const int i = j * PPT + k;
          if (defer && pg0 + i == tail) {
            deferred_tile = j;
            deferred_k = k;
            continue;
          }
          bulk_g2s_hint(ring + (size_t)s * STAGE + (size_t)k * BLOCK,
                        pool_l + ((size_t)pid_s[i] * g.Hkv + kvh) * BLOCK, (uint32_t)BLOCK, &full[s], policy);
        }
      };
      const int first = min(NS, ntiles);
      for (int j = 0; j < first; ++j) arm(j, true);
      pdl_wait();  // the preceding grid may still be writing the tail page (fused step)
      if (deferred_tile >= 0) {
        const int s = deferred_tile % NS, i = deferred_tile * PPT + deferred_k;
        bulk_g2s_hint(ring + (size_t)s * STAGE + (size_t)deferred_k * BLOCK,
                      pool_l + ((size_t)pid_s[i] * g.Hkv + kvh) * BLOCK, (uint32_t)BLOCK, &full[s], policy);
      }
      const uint32_t idesc = idesc_f16_f32(128, 16);
      const uint32_t bq_addr = smem_u32(bq);
      int i = 0, jr = first;  // next QK tile, next refill tile
      uint64_t t0 = globaltimer_ns();
      while (i < ntiles || jr < ntiles) {
        bool prog = false;
        if (i < ntiles && mbar_try_wait(&a_full[i & 1], (i >> 1) & 1) &&
            (i < 2 || mbar_try_wait(&s_empty[i & 1], ((i - 2) >> 1) & 1))) {
          tc_fence_after();
          const uint32_t a_base = tmem + C::TM_A + (uint32_t)((i & 1) * C::ACOLS);
          const uint32_t d_base = tmem + C::TM_S + (uint32_t)((i & 1) * SCOLS);
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const int wdw = (ks >> 1) / GPW;
            const uint64_t bdesc =
                smem_desc_sw128(bq_addr + (uint32_t)((ks >> 2) * SCOLS * 128 + wdw * 16 * 128 + (ks & 3) * 32));
            tc_mma_ts(d_base + (uint32_t)(16 * wdw), a_base + (uint32_t)(8 * ks), bdesc, idesc,
                      (ks % (2 * GPW)) != 0 ? 1u : 0u);
          }
          tc_commit(&qk_done[i & 1]);
          ++i;
          prog = true;
        }
        if (jr < ntiles && mbar_try_wait(&empty[jr % NS], ((jr - NS) / NS) & 1)) {
          fence_proxy_async_smem();
          arm(jr, false);
          ++jr;
          prog = true;
        }
        if (*abort_s) break;
        if (prog) {
          t0 = globaltimer_ns();
        } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
          flag_error(a.status, kDevTimeout);
          *abort_s = 1;
          break;
        }
      }
      if (*abort_s) {
        // drain: the MMAs issued and the copies in flight, each wait bounded
        if (i > 0) (void)mbar_wait_bounded(&qk_done[(i - 1) & 1], ((i - 1) >> 1) & 1, nullptr);
        for (int j = max(0, jr - NS); j < jr; ++j) (void)mbar_wait_bounded(&full[j % NS], (j / NS) & 1, nullptr);
      }
    }
    __syncwarp();
  } else if (warp < kTokWarps) {
    // =============================== token warps
    const int t = tid;  // token of the tile, TMEM lane t
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    pdl_wait();  // the query operands come from the preceding grid
    // query-side constants: score = F_h (sum_g S_g (hi_g,h + lo_g,h) + Z_g Qs_h,g)
    const float* aux_base = ws.qaux + ((size_t)b * g.Hq + (size_t)kvh * GQ) * 8;
    // Qs_h,g: in registers up to four heads; with eight heads in shared memory ([g][h], read
    // as broadcast vectors), since the 13-warp CTA allocates registers as 16 warps (128 each)
    constexpr bool QS_SMEM = GQ == 8;
    float F[GQ], Qs[QS_SMEM ? 1 : GQ][GROUPS];
    float* qs_s = reinterpret_cast<float*>(smem + C::M_QS);
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      const float inv = aux_base[h * 8];  // 2^-e_h
      F[h] = inv * ldexpf(sm_log2, -a.k_exp_K);
#pragma unroll
      for (int gg = 0; gg < GROUPS; ++gg) {
        const float v = ldexpf(aux_base[h * 8 + 1 + gg] / inv, a.k_exp_K);
        if constexpr (QS_SMEM) {
          if (t == 0) qs_s[gg * 8 + h] = v;
        } else {
          Qs[h][gg] = v;
        }
      }
    }
    if constexpr (QS_SMEM) bar_sync_named(kBarTok, 128);
    // B of the QK product: row n = (window, group in window, head, hi|lo), K = channels,
    // 128-byte swizzled K-major; 16-byte chunk (n, m) holds channels 8m .. 8m + 7
    for (int c = t; c < SCOLS * (D / 8); c += 128) {
      const int nrow = c / (D / 8), m = c % (D / 8);
      const int wdw = nrow >> 4, lc = nrow & 15;
      const int gl = lc / CG, h = (lc % CG) >> 1, hl = lc & 1;
      const int gg = wdw * GPW + gl;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (gl < GPW && gg < GROUPS && h < GQ && (m >> 2) == gg) {
        const int gid = G8 ? h : 2 * (h & 3) + hl;
        const int plane = G8 ? hl : 0;
        const uint2* f = ws.qfrag + ((((size_t)b * g.Hkv + kvh) * NT + plane) * (D / 16) + (m >> 1)) * 32 + gid * 4;
        uint32_t w4[4];
#pragma unroll
        for (int tg = 0; tg < 4; ++tg) w4[tg] = (m & 1) ? f[tg].y : f[tg].x;
        v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      *reinterpret_cast<uint4*>(bq + sw128_offset(nrow, 8 * m, SCOLS)) = v;
    }
    fence_proxy_async_smem();  // the tensor core reads it through the async proxy

    // K codes of token t of tile j -> A operand in TMEM buffer j & 1
    auto unpack = [&](int j) -> bool {
      const int s = j % NS;
      if (!mbar_wait_bounded(&full[s], (j / NS) & 1, a.status)) return false;
      const uint8_t* krow = ring + (size_t)s * STAGE + (t >> lgP) * BLOCK + (t & (P - 1)) * ROW;
      uint32_t kw[D / 16];
#pragma unroll
      for (int v = 0; v < D / 64; ++v) {
        const uint4 q4 = *reinterpret_cast<const uint4*>(krow + 16 * v);
        kw[4 * v] = q4.x; kw[4 * v + 1] = q4.y; kw[4 * v + 2] = q4.z; kw[4 * v + 3] = q4.w;
      }
      // word tig * (D/64) + w, slot x: channels c, c + 1 with c = 32 gg + 16 kt + 8 hh + 2 tig
      // (gg = (D/64 == 2 ? 2w : 0) + x/4, kt = (x/2)&1, hh = x&1) -> TMEM column 8 (2 gg + kt) + 4 hh + tig,
      // K index = channel.  Columns [32 w, 32 w + 32) come from the words of w: one 32-column store each.
      const uint32_t dst = lane_base + C::TM_A + (uint32_t)((j & 1) * C::ACOLS);
#pragma unroll
      for (int w = 0; w < D / 64; ++w) {
        uint32_t r32[32];
#pragma unroll
        for (int tg = 0; tg < 4; ++tg) {
          const uint32_t wd = kw[tg * (D / 64) + w], w6 = wd >> 6;
#define OSCAR_K_COL(X) r32[8 * (2 * ((X) >> 2) + (((X) >> 1) & 1)) + 4 * ((X) & 1) + tg] = subnormal_slot<X>(wd, w6);
          OSCAR_K_COL(0) OSCAR_K_COL(1) OSCAR_K_COL(2) OSCAR_K_COL(3)
          OSCAR_K_COL(4) OSCAR_K_COL(5) OSCAR_K_COL(6) OSCAR_K_COL(7)
#undef OSCAR_K_COL
        }
        tmem_st32(dst + (uint32_t)(32 * w), r32);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[j & 1]);
      return true;
    };

    float mm[GQ], lsum[GQ];   // reference and weight sums; the rescale threshold is mm + kWeightShift + kRescaleLog2
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      mm[h] = -INFINITY;
      lsum[h] = 0.f;
    }
    const uint32_t k23 = static_cast<uint32_t>(a.k_exp_K + 14) << 23;  // K scales: s * 2^(k_K + 14)
    // this token's slot in the weight operand: block j16, lane (column, tig), word bb, half aa
    const int j16 = t >> 4, t16 = t & 15;
    const int tg = t16 & 3, bb = (t16 >> 2) & 1, aa = t16 >> 3;
    // Every iteration ends with the 128 token threads agreeing (barrier reduction)
    // on whether any of them failed a bounded wait, so that they leave the loop
    // together and never wait on a named barrier the others have left.
    bool okl = unpack(0);
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int bsel = i & 1;
      if (okl && i + 1 < ntiles) okl = unpack(i + 1);
      okl = okl && mbar_wait_bounded(&qk_done[bsel], (i >> 1) & 1, a.status);
      if (bar_red_or(kBarTok, 128, !okl)) { ok = false; break; }
      tc_fence_after();
      // scores: the K (scale, zero) words of this token, then the score windows two at a time
      const int s = i % NS;
      const int blk = t >> lgP;
      const uint8_t* ps = ring + (size_t)s * STAGE + blk * BLOCK + KSZ + (t & (P - 1)) * SZ;
      uint32_t sz[GROUPS];
      if constexpr (D == 128) {
        const uint4 q4 = *reinterpret_cast<const uint4*>(ps);
        sz[0] = q4.x; sz[1] = q4.y; sz[2] = q4.z; sz[3] = q4.w;
      } else {
        const uint2 q2 = *reinterpret_cast<const uint2*>(ps);
        sz[0] = q2.x; sz[1] = q2.y;
      }
      const int tp = (pg0 + i * PPT) * P + t;
      const bool valid = ((pmask_s[s] >> blk) & 1u) && tp >= S && tp < h_end;
      float sc[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) sc[h] = 0.f;
      constexpr int WCH = NWIN > 2 ? 2 : NWIN;
#pragma unroll
      for (int w0 = 0; w0 < NWIN; w0 += WCH) {
        uint32_t sr[WCH][16];
#pragma unroll
        for (int w = 0; w < WCH; ++w)
          tmem_ld16_nowait(lane_base + C::TM_S + (uint32_t)(bsel * SCOLS + 16 * (w0 + w)), sr[w]);
        tmem_wait_ld();
#pragma unroll
        for (int gg = w0 * GPW; gg < (w0 + WCH) * GPW && gg < GROUPS; ++gg) {
          const float Sg = scale_times_pow2(sz[gg], k23), Zg = bf16_hi(sz[gg]);
          float qz[GQ];
          if constexpr (QS_SMEM) {
            const float4 q0 = *reinterpret_cast<const float4*>(qs_s + gg * 8);
            const float4 q1 = *reinterpret_cast<const float4*>(qs_s + gg * 8 + 4);
            qz[0] = q0.x; qz[1] = q0.y; qz[2] = q0.z; qz[3] = q0.w;
            qz[4] = q1.x; qz[5] = q1.y; qz[6] = q1.z; qz[7] = q1.w;
          } else {
#pragma unroll
            for (int h = 0; h < GQ; ++h) qz[h] = Qs[h][gg];
          }
#pragma unroll
          for (int h = 0; h < GQ; ++h) {
            const int col = (gg % GPW) * CG + 2 * h;
            const float d = __uint_as_float(sr[gg / GPW - w0][col]) + __uint_as_float(sr[gg / GPW - w0][col + 1]);
            sc[h] = fmaf(Zg, qz[h], fmaf(Sg, d, sc[h]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[bsel]);
#pragma unroll
      for (int h = 0; h < GQ; ++h) sc[h] = valid ? sc[h] * F[h] : -INFINITY;
      // lazy softmax reference, shared by the CTA: it moves only when a score exceeds it by kRescaleLog2
      bool need = false;
#pragma unroll
      for (int h = 0; h < GQ; ++h) need |= sc[h] > mm[h] + (kWeightShift + kRescaleLog2);
      need = bar_red_or(kBarTok, 128, need);
      float al[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) al[h] = 1.f;
      if (need) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          float m = sc[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) red_s[warp * 8 + h] = m;
        }
        bar_sync_named(kBarTok, 128);
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          const float M = fmaxf(fmaxf(red_s[h], red_s[8 + h]), fmaxf(red_s[16 + h], red_s[24 + h]));
          const float nm = M > mm[h] + (kWeightShift + kRescaleLog2) ? M - kWeightShift : mm[h];
          al[h] = nm == mm[h] ? 1.f : ex2(mm[h] - nm);
          mm[h] = nm;
          lsum[h] *= al[h];
        }
      }
      okl = i < 2 || mbar_wait_bounded(&w_empty[bsel], ((i - 2) >> 1) & 1, a.status);
      if (okl) {
        if (t == 0) {
          flag_s[bsel] = need ? 1 : 0;
#pragma unroll
          for (int h = 0; h < GQ; ++h) alpha_s[bsel * 8 + h] = al[h];
        }
        uint8_t* wb = reinterpret_cast<uint8_t*>(wbuf + (size_t)(bsel * kPvWarps + j16) * NT * 32);
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          const float p = ex2(sc[h] - mm[h]);
          lsum[h] += p;
          const __half hi = __float2half_rn(p);
          const __half lo = __float2half_rn(p - __half2float(hi));
          const int n0 = G8 ? h : 2 * h;
          const int pl1 = G8 ? 1 : 0, n1 = G8 ? h : 2 * h + 1;
          *reinterpret_cast<__half*>(wb + ((0 * 32 + n0 * 4 + tg) * 8 + bb * 4 + aa * 2)) = hi;
          *reinterpret_cast<__half*>(wb + ((pl1 * 32 + n1 * 4 + tg) * 8 + bb * 4 + aa * 2)) = lo;
        }
      }
      if (bar_red_or(kBarTok, 128, !okl)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_full[bsel]);
    }
    if (!ok) *abort_s = 1;
    // finalise: l per head (sum over the CTA's tokens), the reference
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      float l = lsum[h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      lsum[h] = l;
    }
    bar_sync_named(kBarJoin, kTcThreads);  // (1) every role is done with the ring
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < GQ; ++h) lred_s[warp * 8 + h] = lsum[h];
    if (t == 0)
#pragma unroll
      for (int h = 0; h < GQ; ++h) mm_s[h] = mm[h];
  } else {
    // =============================== value warps
    const int pw = warp - kTokWarps;  // 16-token block pw of every tile
    pdl_wait();
    if (do_win && pw < 4)
      window_chunk<D, 128>(a, b, kvh, x, smem + C::WIN, tid - 32 * kTokWarps, [] { bar_sync_named(kBarWin, 128); });
    const int gid = lane >> 2, tig = lane & 3;
    constexpr int NH = G8 ? 2 : 1;
    const int zv = gid & (GROUPS - 1);
    PvLane L;
    L.oV = VC + tig * ROW + (D == 128 ? gid * 4 : (gid >> 1) * 4);
    L.oVs = VSZ + tig * SZ;
    L.oVz = L.oVs + 4 * zv;
    L.psel = (gid & 1) ? 0x7632u : 0x5410u;
    const uint32_t magic = a.code_magic;
    const uint32_t v23 = static_cast<uint32_t>(a.k_exp_V) << 23;
    float acc[MT][4];
    float zacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;
    const int tok0 = 16 * pw;
    const int blk = tok0 >> lgP, slot0 = tok0 & (P - 1);
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int bsel = i & 1, s = i % NS;
      if (!mbar_wait_bounded(&w_full[bsel], (i >> 1) & 1, a.status) ||
          !mbar_wait_bounded(&full[s], (i / NS) & 1, a.status)) {
        ok = false;
        break;
      }
      if (flag_s[bsel]) {  // the reference moved: rescale the accumulators of each head
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          const float al = alpha_s[bsel * 8 + (G8 ? 2 * tig + j : tig)];
          if constexpr (G8) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              acc[mt][j] *= al;
              acc[mt][2 + j] *= al;
            }
            zacc[j] *= al;
            zacc[2 + j] *= al;
          } else {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int r = 0; r < 4; ++r) acc[mt][r] *= al;
#pragma unroll
            for (int r = 0; r < 4; ++r) zacc[r] *= al;
          }
        }
      }
      const int tb = (pg0 + i * PPT) * P + tok0;
      if (((pmask_s[s] >> blk) & 1u) && tb + 16 > S && tb < h_end) {
        const uint8_t* buf = ring + (size_t)s * STAGE + blk * BLOCK;
        const uint2* wf = wbuf + (size_t)(bsel * kPvWarps + pw) * NT * 32;
        if (tb >= S && tb + 16 <= h_end)
          pv_block<D, GQ, true>(L, buf, slot0, tb, wf, acc, zacc, S, h_end, magic, v23, lane);
        else
          pv_block<D, GQ, false>(L, buf, slot0, tb, wf, acc, zacc, S, h_end, magic, v23, lane);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&w_empty[bsel]);
        mbar_arrive(&empty[s]);
      }
    }
    if (!ok) *abort_s = 1;
    bar_sync_named(kBarJoin, kTcThreads);  // (1) every role is done with the ring
    // this warp's share in real units: channel 16 mt + gid (+ 8) sits in slot (2 mt) mod 8 (+ 1)
    // of its half-word (code scale 2^(slot_pos - 10)); the zero term of group mt / 2
    float zs[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) zs[j] = G8 ? zacc[j] : zacc[0] + zacc[1];
    float zg[NH][GROUPS];
#pragma unroll
    for (int j = 0; j < NH; ++j)
#pragma unroll
      for (int gi = 0; gi < GROUPS; ++gi) zg[j][gi] = __shfl_sync(0xffffffffu, zs[j], gi * 4 + tig);
    float* mrg = reinterpret_cast<float*>(ring);  // [kPvWarps][8][D]
    const float vscale = ldexpf(1.f, -a.k_exp_V);
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      const int hh = G8 ? 2 * tig + j : tig;
      if (hh < GQ) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int ch_a = 16 * mt + gid, ch_b = ch_a + 8;
          const float va_ = G8 ? acc[mt][j] : acc[mt][0] + acc[mt][1];
          const float vb_ = G8 ? acc[mt][2 + j] : acc[mt][2] + acc[mt][3];
          const float za = zg[j][mt >> 1] * vscale;
          const float pa_ = static_cast<float>(1 << (10 - slot_pos((2 * mt) & 7)));
          const float pb_ = static_cast<float>(1 << (10 - slot_pos((2 * mt + 1) & 7)));
          mrg[(pw * 8 + hh) * D + ch_a] = fmaf(va_, vscale * pa_, za);
          mrg[(pw * 8 + hh) * D + ch_b] = fmaf(vb_, vscale * pb_, za);
        }
      }
    }
  }
  if (warp == kCtrlWarp) bar_sync_named(kBarJoin, kTcThreads);  // (1)
  pdl_launch_dependents();
  __syncthreads();  // (2) shares and sums in shared memory
  if (!*abort_s) {
    const float* mrg = reinterpret_cast<const float*>(ring);
    const int stride = a.wl.win_chunks + a.wl.max_splits;
    for (int idx = tid; idx < GQ * D; idx += kTcThreads) {
      const int hh = idx / D, ch = idx % D;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kPvWarps; ++w) v += mrg[(w * 8 + hh) * D + ch];
      float* pp = ws.part + (((size_t)b * g.Hq + (size_t)kvh * GQ + hh) * stride + a.wl.win_chunks + x) * (D + 4);
      pp[4 + ch] = v;
      if (ch == 0) {
        pp[0] = mm_s[hh];
        pp[1] = (lred_s[hh] + lred_s[8 + hh]) + (lred_s[16 + hh] + lred_s[24 + hh]);
      }
    }
  }
  __syncthreads();  // (3)
  if (warp == kCtrlWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int D, int GQ>
int launch_tc_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  using C = TcCfg<D, GQ>;
  const size_t smem = C::smem_bytes(a.wl.tc_stages);
  auto kern = decode_tc_kernel<D, GQ>;
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.wl.tc_grid_x, a.g.Hkv, a.batch);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return (int)cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D>
int launch_tc_d(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  switch (a.g.gq()) {
    case 1: return launch_tc_t<D, 1>(a, s, pdl);
    case 2: return launch_tc_t<D, 2>(a, s, pdl);
    case 4: return launch_tc_t<D, 4>(a, s, pdl);
    default: return launch_tc_t<D, 8>(a, s, pdl);
  }
}

}  // namespace

size_t decode_tc_smem_bytes(int head_dim, int gq, int stages) {
  if (head_dim == 128) {
    switch (gq) {
      case 1: return TcCfg<128, 1>::smem_bytes(stages);
      case 2: return TcCfg<128, 2>::smem_bytes(stages);
      case 4: return TcCfg<128, 4>::smem_bytes(stages);
      default: return TcCfg<128, 8>::smem_bytes(stages);
    }
  }
  switch (gq) {
    case 1: return TcCfg<64, 1>::smem_bytes(stages);
    case 2: return TcCfg<64, 2>::smem_bytes(stages);
    case 4: return TcCfg<64, 4>::smem_bytes(stages);
    default: return TcCfg<64, 8>::smem_bytes(stages);
  }
}

int launch_decode_tc(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return a.g.D == 128 ? launch_tc_d<128>(a, s, pdl) : launch_tc_d<64>(a, s, pdl);
}

}  // namespace oscar
