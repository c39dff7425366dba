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
//   q_rotate       q' = q R_K per (request, q head); writes the query-side MMA
//                  fragments (f16 hi/lo split, per-head power-of-two scale),
//                  the group sums Q_g = sum_{j in g} q'_j, and q as float32.
//   decode_splitk  grid (1 + splits, kv heads, requests).  x = 0 is the BF16
//                  window split (CUDA cores, float32); x >= 1 streams a range of
//                  INT2 pages through a 4-stage shared-memory ring filled by
//                  non-multicast bulk copies (one per (page, kv head) block,
//                  mbarrier completion), and runs QK and PV on the tensor cores
//                  with mma.sync m16n8k16:
//                    QK  M = 16 tokens, N = (q head, f16 hi|lo), K = 16 channels,
//                        A = K codes unpacked to c*2^(pos-10) in f16 (exact),
//                        B = q' * 2^(e_h) * 2^(10-pos) split hi/lo; one
//                        accumulator per 32-channel group so the BF16 scale and
//                        zero apply in the float32 epilogue;
//                    PV  M = 16 channels, N = (q head, bf16 hi|lo), K = 16 tokens,
//                        A = V codes unpacked to c*2^(pos-7) in bf16 (exact),
//                        B = p_t * scale_{t,g} split hi/lo; the zero term
//                        sum_t p_t zero_{t,g} accumulates in float32.
//                  Online softmax in the log2 domain with float32 max/sum.
//   decode_combine merges the split partials, applies R_V^T once and divides by l.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

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
constexpr int kStages = 4;
constexpr int kStageTokens = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 1023;  // the host plan never asks for more
constexpr int kWinChunk = 16;     // window slots per window CTA
constexpr int kMaxWinChunks = 32;
constexpr float kRescaleLog2 = 8.f;

// ------------------------------------------------------------------ workspace views
struct WsView {
  uint2* qfrag;   // [B][Hkv][NT][D/16][32]
  float* qaux;    // [B][Hq][8]: [0] = 2^-e_h, [1 + g] = Q_g
  float* qplain;  // [B][Hq][D]
  float* part;    // [B][Hq][win_chunks + max_splits][D + 4]: [0] m (log2 domain), [1] l, [4..] acc
};

__device__ __forceinline__ WsView ws_view(const DecodeArgs& a) {
  WsView v;
  v.qfrag = reinterpret_cast<uint2*>(a.ws + a.wl.qfrag_off);
  v.qaux = reinterpret_cast<float*>(a.ws + a.wl.qaux_off);
  v.qplain = reinterpret_cast<float*>(a.ws + a.wl.qplain_off);
  v.part = reinterpret_cast<float*>(a.ws + a.wl.part_off);
  return v;
}

__device__ __forceinline__ float load_q(const DecodeArgs& a, size_t idx) {
  if (a.q_dtype == kDtypeBF16) {
    const uint16_t v = static_cast<const uint16_t*>(a.q)[idx];
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  return static_cast<const float*>(a.q)[idx];
}

// Number of INT2 splits request b needs (0 if it has no history).
__device__ __forceinline__ int splits_for(const DecodeArgs& a, int n) {
  const int h_end = n - a.g.W;
  if (h_end <= a.g.S) return 0;
  const int pages = (h_end - 1) / a.g.P + 1;
  return (pages + a.wl.pages_per_split - 1) / a.wl.pages_per_split;
}

__device__ __forceinline__ bool seq_len_ok(const DecodeArgs& a, int n) {
  return n >= 0 && n <= a.max_seq && n <= a.g.max_pages_per_req * a.g.P;
}

// ------------------------------------------------------------------ q rotate
// grid (Hkv * D/32, B), block 128.  CTA (kvh, grp) computes the 32 rotated
// channels of group grp, q'_j = sum_i q_i R_K[i][j] for j in [32 grp, 32 grp + 32),
// for every query head of kv head kvh, and writes the group sum Q_g and the
// query-side MMA fragments of its two k-tiles.  The power-of-two scale of head
// h is set from ||q_h||_2, which bounds |q'_h|_inf (R_K is orthogonal), so the
// CTAs of a head need not agree on a maximum.
template <int D>
__global__ void __launch_bounds__(kThreads) q_rotate_kernel(DecodeArgs a) {
  pdl_launch_dependents();
  __shared__ __align__(16) float Rs[D][33];   // R_K[:, 32 grp + c], padded
  __shared__ float qs[8][D];
  __shared__ float qr[8][32];
  __shared__ float nrm[8];
  const Geom& g = a.g;
  const int grp = blockIdx.x % (D / 32), kvh = blockIdx.x / (D / 32), b = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int gq = g.gq();
  WsView ws = ws_view(a);
  // R_K column slice: D rows x 32 floats (8 float4 per row), 16-byte loads, all in flight
  {
    const float4* Rg = reinterpret_cast<const float4*>(a.R_K);
    float4 v[D * 8 / kThreads];
#pragma unroll
    for (int u = 0; u < D * 8 / kThreads; ++u) {
      const int idx = t + u * kThreads;  // row idx / 8, float4 idx % 8
      v[u] = __ldg(Rg + (size_t)(idx >> 3) * (D / 4) + grp * 8 + (idx & 7));
    }
#pragma unroll
    for (int u = 0; u < D * 8 / kThreads; ++u) {
      const int idx = t + u * kThreads;
      float* dst = &Rs[idx >> 3][(idx & 7) * 4];
      dst[0] = v[u].x; dst[1] = v[u].y; dst[2] = v[u].z; dst[3] = v[u].w;
    }
  }
  const size_t qbase = ((size_t)b * g.Hq + (size_t)kvh * gq) * D;
  for (int i = t; i < gq * D; i += kThreads) {
    const float x = load_q(a, qbase + i);
    qs[i / D][i % D] = x;
    if (grp == 0) ws.qplain[qbase + i] = x;
  }
  __syncthreads();
  // squared norms: warp w sums heads w, w + 4
  for (int hh = warp; hh < gq; hh += kThreads / 32) {
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss = fmaf(qs[hh][i], qs[hh][i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) nrm[hh] = sqrtf(ss);
  }
  // rotation: lane = channel 32 grp + lane, warp w handles heads w, w + 4
  for (int hh = warp; hh < gq; hh += kThreads / 32) {
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc = fmaf(qs[hh][i], Rs[i][lane], acc);
    qr[hh][lane] = acc;
    float gs = acc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
    if (lane == 0) ws.qaux[((size_t)b * g.Hq + (size_t)kvh * gq + hh) * 8 + 1 + grp] = gs;
  }
  __syncthreads();
  // fragments of the two k-tiles of this group: 8 lanes x 2 k-tiles per head
  for (int idx = t; idx < gq * 16; idx += kThreads) {
    const int hh = idx >> 4, sub = idx & 15;
    const int kt = sub >> 3, hl = (sub >> 2) & 1, tig = sub & 3;
    int e = 0;
    const float mx = nrm[hh];
    if (mx > 0.f) {
      int E;
      frexpf(mx, &E);  // |q'|_inf <= ||q||_2 = mx * (1 + rounding) < 2^E
      e = 5 - E;       // |q'| * 2^e < 32: times 2^(10-pos) <= 1024 stays below the f16 maximum
    }
    if (grp == 0 && sub == 0) ws.qaux[((size_t)b * g.Hq + (size_t)kvh * gq + hh) * 8] = ldexpf(1.f, -e);
    const bool g8 = gq == 8;
    const int gid = g8 ? hh : 2 * (hh & 3) + hl;
    const int plane = g8 ? hl : 0;
    const int ln = gid * 4 + tig;
    const int kk = 2 * grp + kt;
    const int p8 = 4 * grp + 2 * kt;
    uint32_t regs[2];
#pragma unroll
    for (int hpair = 0; hpair < 2; ++hpair) {
      const int ch = 16 * kt + 8 * hpair + 2 * tig;  // channel within the group
      const int pos = slot_pos((p8 + hpair) & 7);
      float v[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float x = ldexpf(qr[hh][ch + u], e + 10 - pos);
        const __half hi = __float2half_rn(x);
        const float lo = x - __half2float(hi);
        v[u] = hl ? lo : __half2float(hi);
      }
      regs[hpair] = pack_half2(v[0], v[1]);
    }
    const size_t fidx = ((((size_t)b * g.Hkv + kvh) * a.wl.nt + plane) * (D / 16) + kk) * 32 + ln;
    ws.qfrag[fidx] = make_uint2(regs[0], regs[1]);
  }
}

// ------------------------------------------------------------------ window chunks (BF16, float32 math)
// The S + W window slots of a (request, kv head) are split into chunks of
// kWinChunk = 16 slots, one CTA each (grid.x < win_chunks).  The chunk's K and
// V rows are staged in shared memory; warp w handles query heads w, w + 4.
// Lane l owns channels [l*D/32, (l+1)*D/32): per token it forms a partial dot
// product, and a 31-shuffle reduction leaves the score of slot l in lane l
// (lanes 16..31 hold copies and are masked out).  Output: one partial (m, l, acc) per (query head, chunk) in the plain
// basis.
template <int D>
__device__ void window_chunk(const DecodeArgs& a, int b, int kvh, int chunk, uint8_t* smem) {
  constexpr int C = D / 32;
  const Geom& g = a.g;
  const int gq = g.gq();
  const int n = a.seq_lens[b];
  const int win = g.window();
  const int t0 = chunk * kWinChunk;
  const int cnt = min(kWinChunk, win - t0);
  uint16_t* ks = reinterpret_cast<uint16_t*>(smem);            // [kWinChunk][D]
  uint16_t* vs = ks + kWinChunk * D;                            // [kWinChunk][D]
  float* qsm = reinterpret_cast<float*>(vs + kWinChunk * D);    // [gq][D]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t sbase = ((size_t)a.layer * g.max_req + a.req_slot[b]) * g.slab_req_elems();
  const uint16_t* kwin = a.slab + sbase + ((size_t)kvh * 2 + 0) * win * D + (size_t)t0 * D;
  const uint16_t* vwin = a.slab + sbase + ((size_t)kvh * 2 + 1) * win * D + (size_t)t0 * D;
  const int nvec = cnt * D / 8;  // 16-byte vectors of 8 bf16
  for (int i = tid; i < nvec; i += kThreads) {
    reinterpret_cast<uint4*>(ks)[i] = reinterpret_cast<const uint4*>(kwin)[i];
    reinterpret_cast<uint4*>(vs)[i] = reinterpret_cast<const uint4*>(vwin)[i];
  }
  WsView ws = ws_view(a);
  for (int i = tid; i < gq * D; i += kThreads) qsm[i] = ws.qplain[((size_t)b * g.Hq + (size_t)kvh * gq) * D + i];
  __syncthreads();
  const int n_recent = n > g.S ? min(n - g.S, g.W) : 0;
  const int slot = t0 + lane;
  const bool valid = lane < cnt && (slot < g.S ? slot < n : (slot - g.S) < n_recent);
  const float sm = kLog2e * rsqrtf((float)D);
  const int stride = a.wl.win_chunks + a.wl.max_splits;
  for (int hh = warp; hh < gq; hh += kThreads / 32) {
    float qv[C];
#pragma unroll
    for (int c = 0; c < C; ++c) qv[c] = qsm[hh * D + lane * C + c];
    float part[kWinChunk];
#pragma unroll
    for (int t = 0; t < kWinChunk; ++t) {
      float dot = 0.f;
      if (t < cnt) {
        const uint16_t* kr = ks + t * D + lane * C;
        if constexpr (C == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(kr);
          dot = fmaf(qv[0], bf16_lo(w.x), dot);
          dot = fmaf(qv[1], bf16_hi(w.x), dot);
          dot = fmaf(qv[2], bf16_lo(w.y), dot);
          dot = fmaf(qv[3], bf16_hi(w.y), dot);
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(kr);
          dot = fmaf(qv[0], bf16_lo(w), dot);
          dot = fmaf(qv[1], bf16_hi(w), dot);
        }
      }
      part[t] = dot;
    }
    // fold the two half-warps, then a transpose-reduction: after the step with
    // offset o a lane keeps the o values of its half; finally part[0] of lane l
    // (and of lane l + 16) is the full dot product of slot l
#pragma unroll
    for (int t = 0; t < kWinChunk; ++t) part[t] += __shfl_xor_sync(0xffffffffu, part[t], 16);
#pragma unroll
    for (int o = kWinChunk / 2; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = upper ? part[i] : part[i + o];
        const float keep = upper ? part[i + o] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const float sc = valid ? part[0] * sm : -INFINITY;
    float m = sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p = (sc == -INFINITY) ? 0.f : ex2(sc - m);
    float l = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    for (int t = 0; t < cnt; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      if (pt != 0.f) {  // warp-uniform
        const uint16_t* vr = vs + t * D + lane * C;
#pragma unroll
        for (int c = 0; c < C; ++c)
          acc[c] = fmaf(pt, __uint_as_float(static_cast<uint32_t>(vr[c]) << 16), acc[c]);
      }
    }
    float* pp = ws.part + (((size_t)b * g.Hq + (size_t)kvh * gq + hh) * stride + chunk) * (D + 4);
#pragma unroll
    for (int c = 0; c < C; ++c) pp[4 + lane * C + c] = acc[c];
    if (lane == 0) {
      pp[0] = m;
      pp[1] = l;
    }
  }
}

// ------------------------------------------------------------------ INT2 split
template <int D, int NT, int P>
struct Int2Layout {
  static constexpr int ROW = D / 4;
  static constexpr int SZ = D / 8;
  static constexpr int KSZ = P * ROW;
  static constexpr int VC = KSZ + P * SZ;
  static constexpr int VSZ = VC + P * ROW;
  static constexpr int BLOCK = VSZ + P * SZ;
  static constexpr int PPS = kStageTokens / P;  // pages per stage
  static constexpr int STAGE = PPS * BLOCK;
  static constexpr int GROUPS = D / 32;
  static constexpr int KT = D / 16;             // QK k-tiles
  static constexpr int MT = D / 16;             // PV m-tiles
};

template <int D, int NT, int P>
__global__ void __launch_bounds__(kThreads) decode_splitk_kernel(DecodeArgs a) {
  using Lay = Int2Layout<D, NT, P>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage_buf = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * Lay::STAGE);
  int* stage_valid = reinterpret_cast<int*>(bars + kStages);

  const Geom& g = a.g;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int gq = g.gq();
  const int n = a.seq_lens[b];
  if (!seq_len_ok(a, n)) {
    if (tid == 0 && blockIdx.x == 0) flag_error(a.status, kDevBadLen);
    pdl_launch_dependents();
    return;
  }
  if ((int)blockIdx.x < a.wl.win_chunks) {
    const int req = a.req_slot[b];
    if (req < 0 || req >= g.max_req) {
      if (tid == 0 && blockIdx.x == 0) flag_error(a.status, kDevBadSlot);
      pdl_launch_dependents();
      return;
    }
    pdl_wait();
    window_chunk<D>(a, b, kvh, blockIdx.x, smem);
    pdl_launch_dependents();
    return;
  }
  const int split = blockIdx.x - a.wl.win_chunks;
  const int h_end = n - g.W;
  if (h_end <= g.S) { pdl_launch_dependents(); return; }
  const int n_hist_pages = (h_end - 1) / P + 1;
  const int pg0 = split * a.wl.pages_per_split;
  if (pg0 >= n_hist_pages) { pdl_launch_dependents(); return; }
  const int pg1 = min(pg0 + a.wl.pages_per_split, n_hist_pages);
  const int n_iters = (pg1 - pg0 + Lay::PPS - 1) / Lay::PPS;

  const int* bt = a.block_table + (size_t)b * a.bt_stride;
  const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int it) {
    const int s = it % kStages;
    uint32_t bytes = 0;
    int mask = 0;
    int pages[Lay::PPS];
#pragma unroll
    for (int i = 0; i < Lay::PPS; ++i) {
      const int lp = pg0 + it * Lay::PPS + i;
      pages[i] = -1;
      if (lp < pg1) {
        const int pid = (lp < a.bt_stride && lp < g.max_pages_per_req) ? bt[lp] : -1;
        if (pid >= 0 && pid < g.num_pages) {
          pages[i] = pid;
          bytes += Lay::BLOCK;
          mask |= 1 << i;
        } else {
          flag_error(a.status, kDevBadPage);
        }
      }
    }
    stage_valid[s] = mask;
    mbar_arrive_expect_tx(&bars[s], bytes);
#pragma unroll
    for (int i = 0; i < Lay::PPS; ++i) {
      if (pages[i] >= 0) {
        const uint8_t* src = pool_l + ((size_t)pages[i] * g.Hkv + kvh) * Lay::BLOCK;
        bulk_g2s(stage_buf + s * Lay::STAGE + i * Lay::BLOCK, src, Lay::BLOCK, &bars[s]);
      }
    }
  };

  if (tid == 0) {
    for (int it = 0; it < kStages && it < n_iters; ++it) issue(it);
  }

  // query side (written by q_rotate): wait for the previous grid
  pdl_wait();
  WsView ws = ws_view(a);
  // Column layout of the MMAs (see q_rotate):
  //  G8 (8 query heads per kv head): columns are heads; the f16 (QK) / bf16 (PV)
  //     hi and lo parts are separate operand planes accumulated into the same
  //     registers.  A lane owns heads 2*tig and 2*tig + 1.
  //  otherwise (<= 4 heads): QK columns are (head, hi|lo) = 2*head + part; PV
  //     columns are (head, group parity) = 2*head + (g & 1) with hi and lo as two
  //     MMAs.  A lane owns head tig.
  constexpr bool G8 = NT == 2;
  constexpr int NH = G8 ? 2 : 1;  // heads per lane
  uint32_t qb[NT][Lay::KT][2];
  float qscale[NH];
  float qg[NH][Lay::GROUPS];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool col_ok = G8 || (gid >> 1) < gq;
#pragma unroll
    for (int kk = 0; kk < Lay::KT; ++kk) {
      const uint2 f = ws.qfrag[((((size_t)b * g.Hkv + kvh) * NT + nt) * Lay::KT + kk) * 32 + lane];
      qb[nt][kk][0] = col_ok ? f.x : 0u;
      qb[nt][kk][1] = col_ok ? f.y : 0u;
    }
  }
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const int hh = G8 ? 2 * tig + j : tig;
    const float* aux = ws.qaux + ((size_t)b * g.Hq + kvh * gq + min(hh, gq - 1)) * 8;
    qscale[j] = hh < gq ? aux[0] : 0.f;
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) qg[j][gi] = hh < gq ? aux[1 + gi] : 0.f;
  }

  const float sm_log2 = kLog2e * rsqrtf((float)D);
  float m_run[NH], l_run[NH];
  float acc[Lay::MT][4];
  float zacc[NH][Lay::GROUPS];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) zacc[j][gi] = 0.f;
  }
#pragma unroll
  for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;

  // rows of this lane inside a 16-token block (token order sigma(k) = k/2 + 8*(k%2))
  const int ra = (gid >> 1) + 8 * (gid & 1);      // sigma(gid)
  const int rb = 4 + (gid >> 1) + 8 * (gid & 1);  // sigma(gid + 8)
  const int w_off = 16 * warp;                    // this warp's block inside the stage
  const int pi = w_off / P, slot0 = w_off % P;

  bool aborted = false;
  int it_fail = 0;
  for (int it = 0; it < n_iters; ++it) {
    const int s = it % kStages;
    const bool ok = mbar_wait_bounded(&bars[s], (it / kStages) & 1, a.status);
    if (ok) {
      const int valid_mask = stage_valid[s];
      const bool page_ok = (valid_mask >> pi) & 1;
      const int tb = (pg0 + it * Lay::PPS) * P + w_off;  // absolute token of row 0 of the block
      const uint8_t* buf = stage_buf + s * Lay::STAGE + pi * Lay::BLOCK;
      // ---------------- QK
      uint32_t ua[D / 8], ub[D / 8];  // f16 code pairs of rows ra and rb
      {
        const uint8_t* kc = buf;
        if constexpr (D == 128) {
          const uint2 wa = *reinterpret_cast<const uint2*>(kc + (slot0 + ra) * Lay::ROW + tig * 8);
          const uint2 wb = *reinterpret_cast<const uint2*>(kc + (slot0 + rb) * Lay::ROW + tig * 8);
          uint32_t t8[8];
          unpack_word(wa.x, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ua[x] = t8[x];
          unpack_word(wa.y, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ua[8 + x] = t8[x];
          unpack_word(wb.x, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ub[x] = t8[x];
          unpack_word(wb.y, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ub[8 + x] = t8[x];
        } else {
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(kc + (slot0 + ra) * Lay::ROW + tig * 4);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(kc + (slot0 + rb) * Lay::ROW + tig * 4);
          unpack_word(wa, ua);
          unpack_word(wb, ub);
        }
      }
      float sc[NH][2];  // scores (log2 domain) of this lane's heads for rows ra, rb
      {
        uint32_t sza[Lay::GROUPS], szb[Lay::GROUPS];
        if constexpr (Lay::GROUPS == 4) {
          const uint4 A4 = *reinterpret_cast<const uint4*>(buf + Lay::KSZ + (slot0 + ra) * Lay::SZ);
          const uint4 B4 = *reinterpret_cast<const uint4*>(buf + Lay::KSZ + (slot0 + rb) * Lay::SZ);
          sza[0] = A4.x; sza[1] = A4.y; sza[2] = A4.z; sza[3] = A4.w;
          szb[0] = B4.x; szb[1] = B4.y; szb[2] = B4.z; szb[3] = B4.w;
        } else {
          const uint2 A2 = *reinterpret_cast<const uint2*>(buf + Lay::KSZ + (slot0 + ra) * Lay::SZ);
          const uint2 B2 = *reinterpret_cast<const uint2*>(buf + Lay::KSZ + (slot0 + rb) * Lay::SZ);
          sza[0] = A2.x; sza[1] = A2.y;
          szb[0] = B2.x; szb[1] = B2.y;
        }
        float dsum[NH][2], zsum[NH][2];
#pragma unroll
        for (int j = 0; j < NH; ++j) dsum[j][0] = dsum[j][1] = zsum[j][0] = zsum[j][1] = 0.f;
#pragma unroll
        for (int gi = 0; gi < Lay::GROUPS; ++gi) {
          float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kt = 0; kt < 2; ++kt) {
            const int p8 = 4 * gi + 2 * kt;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16(c, ua[p8], ub[p8], ua[p8 + 1], ub[p8 + 1], qb[nt][2 * gi + kt][0], qb[nt][2 * gi + kt][1]);
          }
          const float s_a = bf16_lo(sza[gi]), s_b = bf16_lo(szb[gi]);
          const float z_a = bf16_hi(sza[gi]), z_b = bf16_hi(szb[gi]);
          if constexpr (G8) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              dsum[j][0] = fmaf(s_a, c[j], dsum[j][0]);
              dsum[j][1] = fmaf(s_b, c[2 + j], dsum[j][1]);
              zsum[j][0] = fmaf(z_a, qg[j][gi], zsum[j][0]);
              zsum[j][1] = fmaf(z_b, qg[j][gi], zsum[j][1]);
            }
          } else {
            dsum[0][0] = fmaf(s_a, c[0] + c[1], dsum[0][0]);
            dsum[0][1] = fmaf(s_b, c[2] + c[3], dsum[0][1]);
            zsum[0][0] = fmaf(z_a, qg[0][gi], zsum[0][0]);
            zsum[0][1] = fmaf(z_b, qg[0][gi], zsum[0][1]);
          }
        }
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          sc[j][0] = fmaf(dsum[j][0], qscale[j], zsum[j][0]) * sm_log2;
          sc[j][1] = fmaf(dsum[j][1], qscale[j], zsum[j][1]) * sm_log2;
        }
      }
      const int ta = tb + ra, tbk = tb + rb;
      // every row of the block is a history token on a mapped page (warp-uniform)
      const bool full_block = page_ok && tb >= g.S && tb + 15 < h_end;
      const bool va = page_ok && ta >= g.S && ta < h_end;
      const bool vb = page_ok && tbk >= g.S && tbk < h_end;
      // ---------------- online softmax (per head: lanes sharing tig).  The running
      // reference m_run only moves when a block maximum exceeds it by more than
      // 2^kRescaleLog2, so the accumulators are rescaled rarely; p stays below
      // 2^kRescaleLog2, which float32 sums and bf16 operands absorb.
      float pa[NH], pb[NH];
      float alpha[NH];
      bool rescale = false;
#pragma unroll
      for (int j = 0; j < NH; ++j) {
        const float s_a = va ? sc[j][0] : -INFINITY;
        const float s_b = vb ? sc[j][1] : -INFINITY;
        float mb = fmaxf(s_a, s_b);
        mb = warp_max_xor(mb, 4);
        mb = warp_max_xor(mb, 8);
        mb = warp_max_xor(mb, 16);
        const float m_ref = (mb > m_run[j] + kRescaleLog2) ? mb : m_run[j];
        alpha[j] = 1.f;
        if (m_ref != m_run[j]) {
          alpha[j] = (m_run[j] == -INFINITY) ? 0.f : ex2(m_run[j] - m_ref);
          rescale = true;
          m_run[j] = m_ref;
        }
        pa[j] = (s_a == -INFINITY) ? 0.f : ex2(s_a - m_run[j]);
        pb[j] = (s_b == -INFINITY) ? 0.f : ex2(s_b - m_run[j]);
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          l_run[j] *= alpha[j];
#pragma unroll
          for (int gi = 0; gi < Lay::GROUPS; ++gi) zacc[j][gi] *= alpha[j];
        }
#pragma unroll
        for (int mt = 0; mt < Lay::MT; ++mt) {
          if constexpr (G8) {
            acc[mt][0] *= alpha[0];
            acc[mt][1] *= alpha[NH - 1];
            acc[mt][2] *= alpha[0];
            acc[mt][3] *= alpha[NH - 1];
          } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mt][r] *= alpha[0];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NH; ++j) l_run[j] += pa[j] + pb[j];
      // ---------------- zero term of the values (rows ra, rb)
      {
        const uint32_t* vszA = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + ra) * Lay::SZ);
        const uint32_t* vszB = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + rb) * Lay::SZ);
#pragma unroll
        for (int gi = 0; gi < Lay::GROUPS; ++gi) {
          const float z_a = bf16_hi(vszA[gi]);
          const float z_b = bf16_hi(vszB[gi]);
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            if (full_block) {
              zacc[j][gi] = fmaf(pb[j], z_b, fmaf(pa[j], z_a, zacc[j][gi]));
            } else {
              if (pa[j] > 0.f) zacc[j][gi] = fmaf(pa[j], z_a, zacc[j][gi]);
              if (pb[j] > 0.f) zacc[j][gi] = fmaf(pb[j], z_b, zacc[j][gi]);
            }
          }
        }
      }
      // ---------------- PV
      {
        // value-side A fragments: rows k in {2tig, 2tig+1, 2tig+8, 2tig+9} are tokens
        // sigma(k) = tig, tig+8, tig+4, tig+12; this lane reads word gid (D=128) of each.
        const uint8_t* vc = buf + Lay::VC;
        uint32_t ux[D / 8], uy[D / 8];
        if constexpr (D == 128) {
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig) * Lay::ROW + gid * 4);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 8) * Lay::ROW + gid * 4);
          const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 4) * Lay::ROW + gid * 4);
          const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 12) * Lay::ROW + gid * 4);
          uint32_t t8[8];
          unpack_word_bf16(prmt(w0, w1, 0x5410), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ux[x] = t8[x];
          unpack_word_bf16(prmt(w0, w1, 0x7632), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ux[8 + x] = t8[x];
          unpack_word_bf16(prmt(w8, w9, 0x5410), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) uy[x] = t8[x];
          unpack_word_bf16(prmt(w8, w9, 0x7632), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) uy[8 + x] = t8[x];
        } else {
          const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
          const int wo = (gid >> 1) * 4;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig) * Lay::ROW + wo);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 8) * Lay::ROW + wo);
          const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 4) * Lay::ROW + wo);
          const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 12) * Lay::ROW + wo);
          unpack_word_bf16(prmt(w0, w1, sel), ux);
          unpack_word_bf16(prmt(w8, w9, sel), uy);
        }
        // scales of rows 2tig, 2tig+1, 2tig+8, 2tig+9 (tokens tig, tig+8, tig+4, tig+12)
        const uint32_t* vsr[4] = {
            reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig) * Lay::SZ),
            reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 8) * Lay::SZ),
            reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 4) * Lay::SZ),
            reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 12) * Lay::SZ)};
        // p of this lane's column head at rows 2tig, 2tig+1, 2tig+8, 2tig+9
        const int src0 = (2 * tig) * 4 + (gid >> 1);
        const int src1 = (2 * tig + 1) * 4 + (gid >> 1);
        float pr[4];
        if constexpr (G8) {
          // column head gid lives in lane group tig = gid >> 1 as its head j = gid & 1
          const bool second = (gid & 1) != 0;
          const float a0 = __shfl_sync(0xffffffffu, pa[0], src0), a1 = __shfl_sync(0xffffffffu, pa[NH - 1], src0);
          const float b0 = __shfl_sync(0xffffffffu, pa[0], src1), b1 = __shfl_sync(0xffffffffu, pa[NH - 1], src1);
          const float c0 = __shfl_sync(0xffffffffu, pb[0], src0), c1 = __shfl_sync(0xffffffffu, pb[NH - 1], src0);
          const float d0 = __shfl_sync(0xffffffffu, pb[0], src1), d1 = __shfl_sync(0xffffffffu, pb[NH - 1], src1);
          pr[0] = second ? a1 : a0;
          pr[1] = second ? b1 : b0;
          pr[2] = second ? c1 : c0;
          pr[3] = second ? d1 : d0;
        } else {
          pr[0] = __shfl_sync(0xffffffffu, pa[0], src0);
          pr[1] = __shfl_sync(0xffffffffu, pa[0], src1);
          pr[2] = __shfl_sync(0xffffffffu, pb[0], src0);
          pr[3] = __shfl_sync(0xffffffffu, pb[0], src1);
        }
        // B operands: weights w = p * scale_g, split as hi = bf16 truncation of w and
        // lo = bf16(w - hi) (round to nearest); both go through the MMA into one accumulator
        auto weights = [&](int gi, uint32_t& bh0, uint32_t& bh1, uint32_t& bl0, uint32_t& bl1) {
          float w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            w[u] = pr[u] * bf16_lo(vsr[u][gi]);
            if (!full_block) w[u] = pr[u] > 0.f ? w[u] : 0.f;  // unwritten slots may hold NaN scales
          }
          uint32_t hw[4];
          float lo[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            hw[u] = __float_as_uint(w[u]) & 0xFFFF0000u;
            lo[u] = w[u] - __uint_as_float(hw[u]);
          }
          bh0 = prmt(hw[0], hw[1], 0x7632);
          bh1 = prmt(hw[2], hw[3], 0x7632);
          bl0 = pack_bf162(lo[0], lo[1]);
          bl1 = pack_bf162(lo[2], lo[3]);
        };
        if constexpr (G8) {
#pragma unroll
          for (int gi = 0; gi < Lay::GROUPS; ++gi) {
            uint32_t bh0, bh1, bl0, bl1;
            weights(gi, bh0, bh1, bl0, bl1);
#pragma unroll
            for (int mq = 0; mq < 2; ++mq) {
              const int mt = 2 * gi + mq;
              mma_bf16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bh0, bh1);
              mma_bf16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bl0, bl1);
            }
          }
        } else {
          // column (head, parity): parity gid & 1 selects group 2*gp + parity of pair gp
#pragma unroll
          for (int gp = 0; gp < (Lay::GROUPS + 1) / 2; ++gp) {
            const int gi = min(2 * gp + (gid & 1), Lay::GROUPS - 1);
            uint32_t bh0, bh1, bl0, bl1;
            weights(gi, bh0, bh1, bl0, bl1);
#pragma unroll
            for (int mq = 0; mq < 4; ++mq) {
              const int mt = 4 * gp + mq;  // m-tiles of groups 2gp, 2gp+1
              if (mt < Lay::MT) {
                mma_bf16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bh0, bh1);
                mma_bf16(acc[mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], bl0, bl1);
              }
            }
          }
        }
      }
    }
    // every warp is done with stage s (uniform abort decision)
    aborted = __syncthreads_or(!ok) != 0;
    if (aborted) {
      it_fail = it;
      break;
    }
    if (tid == 0 && it + kStages < n_iters) issue(it + kStages);
  }
  if (aborted) {
    // drain copies still in flight before the CTA exits, again bounded
    if (tid == 0) {
      const int last = min(n_iters, it_fail + kStages);
      for (int it = it_fail; it < last; ++it) (void)mbar_wait_bounded(&bars[it % kStages], (it / kStages) & 1, nullptr);
    }
    __syncthreads();
    pdl_launch_dependents();
    return;
  }
  pdl_launch_dependents();

  // ---------------- per-warp finalisation
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) {
      zacc[j][gi] += __shfl_xor_sync(0xffffffffu, zacc[j][gi], 4);
      zacc[j][gi] += __shfl_xor_sync(0xffffffffu, zacc[j][gi], 8);
      zacc[j][gi] += __shfl_xor_sync(0xffffffffu, zacc[j][gi], 16);
    }
  }
  // cross-warp merge through shared memory (the stage ring is free now)
  float* wm = reinterpret_cast<float*>(smem);   // [4][8]
  float* wl = wm + 32;                          // [4][8]
  float* wacc = wl + 32;                        // [4][8][D]
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const int hh = G8 ? 2 * tig + j : tig;
    if (hh < gq) {
      if (gid == 0) {
        wm[warp * 8 + hh] = m_run[j];
        wl[warp * 8 + hh] = l_run[j];
      }
#pragma unroll
      for (int mt = 0; mt < Lay::MT; ++mt) {
        const int ch_a = 16 * mt + gid, ch_b = ch_a + 8;
        // G8: registers (0, 2) hold head 2tig, (1, 3) head 2tig+1.  Otherwise the
        // register of the group's parity holds the value (the other is a discarded column).
        const int par = (mt >> 1) & 1;
        const float ra_ = G8 ? acc[mt][j] : acc[mt][par];
        const float rb_ = G8 ? acc[mt][2 + j] : acc[mt][2 + par];
        // channel ch of the V row sits in slot s = (ch mod 64) / 8 with bit position vpos(s)
        const int sa = (ch_a & 63) >> 3, sb = (ch_b & 63) >> 3;
        wacc[(warp * 8 + hh) * D + ch_a] = ldexpf(ra_, 7 - slot_pos_bf16(sa)) + zacc[j][ch_a / 32];
        wacc[(warp * 8 + hh) * D + ch_b] = ldexpf(rb_, 7 - slot_pos_bf16(sb)) + zacc[j][ch_b / 32];
      }
    }
  }
  __syncthreads();
  const int stride = a.wl.win_chunks + a.wl.max_splits;
  for (int idx = tid; idx < gq * D; idx += kThreads) {
    const int hh = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * 8 + hh]);
    float accv = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = wm[w * 8 + hh];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      accv = fmaf(f, wacc[(w * 8 + hh) * D + ch], accv);
      L = fmaf(f, wl[w * 8 + hh], L);
    }
    float* pp = ws.part + (((size_t)b * g.Hq + kvh * gq + hh) * stride + blockIdx.x) * (D + 4);
    pp[4 + ch] = accv;
    if (ch == 0) {
      pp[0] = M;
      pp[1] = L;
    }
  }
}

// ------------------------------------------------------------------ combine
// grid (Hq / hpc, B), block 128.  One CTA handles hpc query heads of one
// request: it merges the window partials (plain basis) and the INT2 partials
// (rotated basis), applies R_V^T once per head, divides by l.  R_V and, when the
// plan says they fit, the heads' partials are staged in shared memory by bulk
// copies; otherwise the partials are read from global memory.
template <int D>
__global__ void __launch_bounds__(kThreads) decode_combine_kernel(DecodeArgs a) {
  constexpr int C = D / 32;
  extern __shared__ __align__(16) float csm[];
  float* Rs = csm;                 // [D][D]
  float* parts = Rs + D * D;       // [hpc][stride][D + 4] when staged
  __shared__ float rot[D];
  __shared__ float rotated_out[D];
  __shared__ float wts[kMaxSplits + kMaxWinChunks];
  __shared__ float s_l;
  __shared__ __align__(8) uint64_t bar;
  const Geom& g = a.g;
  const int hpc = a.wl.combine_hpc;
  const int b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  WsView ws = ws_view(a);
  const int wc = a.wl.win_chunks;
  const int stride = wc + a.wl.max_splits;
  const size_t head_bytes = (size_t)stride * (D + 4) * sizeof(float);
  const int h0 = blockIdx.x * hpc;
  const float* gbase = ws.part + ((size_t)b * g.Hq + h0) * stride * (D + 4);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // R_V does not depend on the previous kernel: start its copy before waiting on it
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar, D * D * sizeof(float) + (a.wl.combine_part_smem ? hpc * head_bytes : 0));
    bulk_g2s(Rs, a.R_V, D * D * sizeof(float), &bar);
  }
  pdl_wait();
  if (tid == 0 && a.wl.combine_part_smem) bulk_g2s(parts, gbase, (uint32_t)(hpc * head_bytes), &bar);
  const int n = a.seq_lens[b];
  const int nsp = seq_len_ok(a, n) ? min(splits_for(a, n), kMaxSplits) : 0;
  const int nslot = wc + nsp;
  if (!mbar_wait_bounded(&bar, 0, a.status)) {
    (void)mbar_wait_bounded(&bar, 0, nullptr);
    return;
  }
  for (int hi = 0; hi < hpc; ++hi) {
    const int h = h0 + hi;
    const float* base = a.wl.combine_part_smem ? parts + (size_t)hi * stride * (D + 4)
                                               : gbase + (size_t)hi * stride * (D + 4);
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
    float plain = 0.f;
    if (tid < D) {
      for (int i = 0; i < wc; ++i) plain = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + tid], plain);
      float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
      int i = wc;
      for (; i + 3 < nslot; i += 4) {
        r0 = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + tid], r0);
        r1 = fmaf(wts[i + 1], base[(size_t)(i + 1) * (D + 4) + 4 + tid], r1);
        r2 = fmaf(wts[i + 2], base[(size_t)(i + 2) * (D + 4) + 4 + tid], r2);
        r3 = fmaf(wts[i + 3], base[(size_t)(i + 3) * (D + 4) + 4 + tid], r3);
      }
      for (; i < nslot; ++i) r0 = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + tid], r0);
      rot[tid] = (r0 + r1) + (r2 + r3);
    }
    __syncthreads();
    // (rot R_V^T)_j = sum_k rot_k R_V[j][k]: warp w handles rows [w*D/4, (w+1)*D/4) in batches of 8
    float rl[C];
#pragma unroll
    for (int c = 0; c < C; ++c) rl[c] = rot[lane * C + c];
    for (int j0 = warp * (D / 4); j0 < (warp + 1) * (D / 4); j0 += 8) {
      float sacc[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float* row = Rs + (j0 + r) * D + lane * C;
        float t = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) t = fmaf(rl[c], row[c], t);
        sacc[r] = t;
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sacc[r] += __shfl_xor_sync(0xffffffffu, sacc[r], o);
        if (lane == r) rotated_out[j0 + r] = sacc[r];
      }
    }
    __syncthreads();
    if (tid < D) {
      const float inv = s_l > 0.f ? 1.f / s_l : 0.f;
      const float o = (plain + rotated_out[tid]) * inv;
      const size_t oi = ((size_t)b * g.Hq + h) * D + tid;
      if (a.out_dtype == kDtypeBF16) {
        __nv_bfloat16 hb = __float2bfloat16_rn(o);
        static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
      } else {
        static_cast<float*>(a.out)[oi] = o;
      }
    }
    __syncthreads();
  }
}

template <int D, int NT, int P>
int launch_splitk_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  using Lay = Int2Layout<D, NT, P>;
  size_t smem = kStages * Lay::STAGE + kStages * 8 + kStages * 4;
  const size_t win_smem = 2 * kWinChunk * D * sizeof(uint16_t) + 8 * D * sizeof(float);
  const size_t merge_smem = (64 + 4 * 8 * D) * sizeof(float);
  if (win_smem > smem) smem = win_smem;
  if (merge_smem > smem) smem = merge_smem;
  smem = (smem + 127) & ~size_t(127);
  auto kern = decode_splitk_kernel<D, NT, P>;
  cudaError_t e = ensure_smem_limit(kern, smem);
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

template <int D, int NT>
int launch_splitk_p(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  switch (a.g.P) {
    case 16: return launch_splitk_t<D, NT, 16>(a, s, pdl);
    case 32: return launch_splitk_t<D, NT, 32>(a, s, pdl);
    default: return launch_splitk_t<D, NT, 64>(a, s, pdl);
  }
}

template <int D>
int launch_q_rotate_t(const DecodeArgs& a, cudaStream_t s) {
  q_rotate_kernel<D><<<dim3(a.g.Hkv * (D / 32), a.batch), kThreads, 0, s>>>(a);
  return (int)cudaGetLastError();
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

int launch_q_rotate(const DecodeArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return a.g.D == 128 ? launch_q_rotate_t<128>(a, s) : launch_q_rotate_t<64>(a, s);
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
  cfg.gridDim = dim3(a.g.Hq / a.wl.combine_hpc, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.dynamicSmemBytes = a.wl.combine_smem;
  cudaError_t e;
  if (a.g.D == 128) {
    if ((e = ensure_smem_limit(decode_combine_kernel<128>, a.wl.combine_smem)) != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, a);
  }
  if ((e = ensure_smem_limit(decode_combine_kernel<64>, a.wl.combine_smem)) != cudaSuccess) return (int)e;
  return (int)cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, a);
}

}  // namespace oscar
