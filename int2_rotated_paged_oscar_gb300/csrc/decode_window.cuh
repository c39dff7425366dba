// Pieces shared by the decode kernels: split bookkeeping and the BF16 window
// chunk (sink + recent tokens, float32 on CUDA cores).  Included inside namespace
// oscar's anonymous namespace, after common.cuh and q_rotate.cuh.
#pragma once

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 1023;  // the host plan never asks for more
constexpr int kWinChunk = 16;     // window slots per window CTA
constexpr int kMaxWinChunks = 32;
constexpr float kRescaleLog2 = 8.f;   // the softmax reference moves when a score exceeds it by more
constexpr float kWeightShift = 6.f;   // weights are 2^(s - mm) with mm = reference - kWeightShift

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

// ------------------------------------------------------------------ window chunks (BF16, float32 math)
// The S + W window slots of a (request, kv head) are split into chunks of
// kWinChunk = 16 slots, one CTA each (grid.x < win_chunks).  TH threads (tid is
// the local index, sync() their barrier) stage the chunk's K and V rows in shared
// memory; warp w handles query heads w, w + TH/32, ...
// Lane l owns channels [l*D/32, (l+1)*D/32): per token it forms a partial dot
// product, and a 31-shuffle reduction leaves the score of slot l in lane l
// (lanes 16..31 hold copies and are masked out).  Output: one partial (m, l, acc) per (query head, chunk) in the plain
// basis.
// Q_INPUT: q is read from the call's input (the one-launch decode, which has no
// q_rotate kernel) instead of the workspace copy q_rotate wrote.
template <int D, int TH, bool Q_INPUT = false, typename Sync>
__device__ void window_chunk(const DecodeArgs& a, int b, int kvh, int chunk, uint8_t* smem, int tid, Sync sync) {
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
  const int warp = tid >> 5, lane = tid & 31;
  const size_t sbase = ((size_t)a.layer * g.max_req + a.req_slot[b]) * g.slab_req_elems();
  const uint16_t* kwin = a.slab + sbase + ((size_t)kvh * 2 + 0) * win * D + (size_t)t0 * D;
  const uint16_t* vwin = a.slab + sbase + ((size_t)kvh * 2 + 1) * win * D + (size_t)t0 * D;
  const int nvec = cnt * D / 8;  // 16-byte vectors of 8 bf16
  for (int i = tid; i < nvec; i += TH) {
    reinterpret_cast<uint4*>(ks)[i] = reinterpret_cast<const uint4*>(kwin)[i];
    reinterpret_cast<uint4*>(vs)[i] = reinterpret_cast<const uint4*>(vwin)[i];
  }
  WsView ws = ws_view(a);
  for (int i = tid; i < gq * D; i += TH)
    qsm[i] = Q_INPUT ? load_q(a, ((size_t)b * g.Hq + (size_t)kvh * gq) * D + i)
                     : ws.qplain[((size_t)b * g.Hq + (size_t)kvh * gq) * D + i];
  sync();
  const int n_recent = n > g.S ? min(n - g.S, g.W) : 0;
  const int slot = t0 + lane;
  const bool valid = lane < cnt && (slot < g.S ? slot < n : (slot - g.S) < n_recent);
  const float sm = kLog2e * rsqrtf((float)D);
  const int stride = a.wl.win_chunks + a.wl.max_splits;
  for (int hh = warp; hh < gq; hh += TH / 32) {
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

