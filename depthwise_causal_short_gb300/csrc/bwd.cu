// bwd.cu -- cconv_bwd and its packed-sequence and multi-problem forms: the backward stream
// plus a deterministic reduction (two kernels).
//
// With z recomputed from x and g = dy * sigmoid(z) * (1 + z * (1 - sigmoid(z))):
//   dx[b,t,d]    = sum_{k<W} w[d,W-1-k] * g[b,t+k,d]     (g = 0 for t+k >= T)
//   dw[d,W-1-k]  = sum_{b,t} g[b,t,d] * x[b,t-k,d]
//   dbias[d]     = sum_{b,t} g[b,t,d]
// Definition: kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py (`_dsilu`,
// `_bwd4`, `cconv_bwd_strip`, `cconv_bwd`).  Kept from that design: one pass over x and dy,
// z recomputed in registers from the same x ring the dw sums need, dx for row t-3 finished
// from a g ring three rows later, a 3-row halo after each range, and a fixed-shape
// reduction of fp32 partials instead of atomics.
//
// GB300 layout: every warp runs its own TMA pipeline over one 128-channel strip of a row
// range (S stages of x and dy tiles on the warp's own mbarriers, issued by lane 0); a CTA is
// SW neighbouring strips x (8 / SW) consecutive ranges.  Arithmetic is packed f32x2, and
// each warp keeps one fp32 partial record ([5][32*VEC]: four lags of dw, then dbias).
// Because each lane owns its channels for the whole range, the time sum needs no shuffles.
// The CTA adds its ranges' records per strip in a fixed order in shared memory; a second
// small kernel adds each channel's records across CTAs in a fixed order, launched as a
// programmatic dependent of the first so that its launch overlaps the stream's tail.
//
// The same body also serves packed sequences (kModeVarlen: sequence boundaries are events
// at single rows, with the initial state's gradient written), no activation (kModeActNone),
// and several problems in one launch (cconv_bwd_multi_kernel).
//
// Rows of 512 channels or more take a lockstep form instead (cconv_bwd_ls_kernel): a
// producer warp loads 8 (from 2048 channels) or 4 neighbouring strips of one row range per
// stage, for x and dy together, and as many consumer warps run the same per-warp tile code
// on their strip of it.
#include <type_traits>

#include "strip.cuh"

namespace cconv {

static __device__ unsigned g_fault_bwd = 0;

int read_clear_fault_bwd(unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbol(out, g_fault_bwd, sizeof(unsigned)) != cudaSuccess) return CCONV_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_fault_bwd, &zero, sizeof(unsigned)) != cudaSuccess) return CCONV_ERR_CUDA;
  return CCONV_OK;
}

constexpr int kRec = 5;  // partial record rows: dw lags 0..3, dbias

struct BwdArgs {
  const void* w;
  const void* bias;
  uint16_t* dx;   // [B,T,D] contiguous bf16 ([total, D] for packed sequences)
  float* ws;      // [grid][SW][kRec][32*VEC] fp32 partial records, one per (CTA, strip)
  int64_t D;
  int T, BT;
  int n_cb, wpc;
  int W, wdt;
  // packed sequences only
  const int32_t* cu;        // [nseq + 1] row offsets
  const uint16_t* init;     // [S, D, W-1] initial states, or null (zeros)
  const int32_t* idx;       // [nseq] slot of each sequence's initial state, or null (slot i)
  int64_t S;                // slots of init (nseq without idx)
  uint16_t* dinit;          // [nseq, D, W-1] gradient of each sequence's initial state, or null
  int nseq;
};

// Slot of sequence i's initial state, or -1 when the index is unusable (negative or >= S:
// the sequence then starts from zeros, and the index check reports it).
__device__ __forceinline__ int64_t init_slot(const BwdArgs& p, int i) {
  const int64_t s = p.idx ? static_cast<int64_t>(p.idx[i]) : i;
  return (s >= 0 && s < p.S) ? s : -1;
}

// Kernel modes: the batched [B,T,D] form with SiLU is mode 0.
enum : int { kModeVarlen = 1, kModeActNone = 2 };

// 2g for one row, from its x and dy and the x ring h = (x[t-1], x[t-2], x[t-3]).  With
// halved taps hz = z / 2 and th = tanh(hz): sigmoid(z) = (1 + th) / 2, 1 - sigmoid(z) =
// (1 - th) / 2, so g = dy sigmoid(z) (1 + z (1 - sigmoid(z))) = dy (1 + th) (1 + hz (1 - th)) / 2.
// The kernel carries g2 = 2g: dx = sum_k (w/2) g2 uses the same halved taps, and the dw / dbias
// sums of g2 are halved once, when the partial record is written.
// Without the activation g = dy, g2 = 2 dy.
template <int P, bool ACT>
__device__ __forceinline__ void bwd_g(const f2 (&x)[P], const f2 (&dy)[P], const f2 (&h)[3][P],
                                      const f2 (&tap)[4][P], const f2 (&bias2)[P], f2 (&g)[P]) {
  const f2 one = f2_splat(1.0f);
  const f2 mone = f2_splat(-1.0f);
  if constexpr (!ACT) {
#pragma unroll
    for (int q = 0; q < P; ++q) g[q] = f2_add(dy[q], dy[q]);
    return;
  }
#pragma unroll
  for (int q = 0; q < P; ++q) {
    f2 hz = f2_fma(tap[0][q], x[q], bias2[q]);
    hz = f2_fma(tap[1][q], h[0][q], hz);
    hz = f2_fma(tap[2][q], h[1][q], hz);
    hz = f2_fma(tap[3][q], h[2][q], hz);
    const f2 th = f2_tanh(hz);
    const f2 d1 = f2_fma(hz, f2_fma(th, mone, one), one);  // 1 + hz (1 - th)
    g[q] = f2_mul(f2_mul(dy[q], f2_add(th, one)), d1);   // dy (1 + th) (1 + hz (1 - th))
  }
}

// dw lags and dbias (of g2 = 2g): acc[k] += g2[t] x[t-k], acc[4] += g2[t]
template <int P>
__device__ __forceinline__ void bwd_acc(const f2 (&x)[P], const f2 (&h)[3][P], const f2 (&g)[P],
                                        f2 (&acc)[kRec][P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    acc[0][q] = f2_fma(g[q], x[q], acc[0][q]);
    acc[1][q] = f2_fma(g[q], h[0][q], acc[1][q]);
    acc[2][q] = f2_fma(g[q], h[1][q], acc[2][q]);
    acc[3][q] = f2_fma(g[q], h[2][q], acc[3][q]);
    acc[4][q] = f2_add(g[q], acc[4][q]);
  }
}

// dx[t-3] = sum_k w[d,W-1-k] g[t-3+k] = sum_k tap[k] g2[t-3+k] (halved taps), from g2[t] and
// the ring gr = (g2[t-1], g2[t-2], g2[t-3])
template <int P>
__device__ __forceinline__ void bwd_dx(const f2 (&g)[P], const f2 (&gr)[3][P],
                                       const f2 (&tap)[4][P], f2 (&dxv)[P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    f2 v = f2_mul(tap[3][q], g[q]);
    v = f2_fma(tap[2][q], gr[0][q], v);
    v = f2_fma(tap[1][q], gr[1][q], v);
    v = f2_fma(tap[0][q], gr[2][q], v);
    dxv[q] = v;
  }
}

template <int P>
__device__ __forceinline__ void rings_push(f2 (&h)[3][P], f2 (&gr)[3][P], const f2 (&x)[P],
                                           const f2 (&g)[P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    h[2][q] = h[1][q];
    h[1][q] = h[0][q];
    h[0][q] = x[q];
    gr[2][q] = gr[1][q];
    gr[1][q] = gr[0][q];
    gr[0][q] = g[q];
  }
}

// Packed sequences: the gradient of initial-state entry j (row ss - (W-1) + j) is the dx
// formula at that row with g = 0 before the sequence; this lane's VEC channels.
template <int VEC>
__device__ __forceinline__ void store_dinit(uint16_t* dinit, int i, int64_t D, int W, int j,
                                            int64_t d0, const f2 (&v)[VEC / 2]) {
  const int L = W - 1;
  uint16_t* o = dinit + (static_cast<int64_t>(i) * D + d0) * L + j;
#pragma unroll
  for (int q = 0; q < VEC / 2; ++q) {
    float lo, hi;
    f2_unpack(v[q], lo, hi);
    o[(2 * q) * L] = f32_to_bf16(lo);
    o[(2 * q + 1) * L] = f32_to_bf16(hi);
  }
}

// Rows of one tile for this lane.  FULL: every row computes g, accumulates dw / dbias and
// stores dx[t-3].  Otherwise rows before `from` were done with the previous tile, rows
// before a only fill the x ring, halo rows after e give g (for the last dx rows) only.
// STORE: this lane's channels exist, so stores need no per-row test.  The dx row pointer
// (row t-3) advances by D per row.
template <int VEC, int R, bool FULL, bool STORE, bool ACT>
__device__ __forceinline__ void bwd_tile(const uint8_t* xt, const uint8_t* dyt, int lane,
                                         const TileCursor& c, bool active, const BwdArgs& p,
                                         int64_t d0, const f2 (&tap)[4][VEC / 2],
                                         const f2 (&bias2)[VEC / 2], f2 (&h)[3][VEC / 2],
                                         f2 (&gr)[3][VEC / 2], f2 (&acc)[kRec][VEC / 2]) {
  constexpr int P = VEC / 2;
  constexpr int ROWB = 32 * VEC * 2;
  uint16_t* dxrow = p.dx + (static_cast<int64_t>(c.b) * p.T + (c.tt - kRing)) * p.D + d0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int t = c.tt + i;
    if (FULL || t >= c.from) {
      f2 x[P], g[P];
      smem_row<VEC>(xt + i * ROWB, lane, x);
      if (FULL || t >= c.a) {
        f2 dy[P];
        smem_row<VEC>(dyt + i * ROWB, lane, dy);
        bwd_g<P, ACT>(x, dy, h, tap, bias2, g);
        if (FULL || t < c.e) bwd_acc<P>(x, h, g, acc);
        if (FULL || (t - kRing >= c.a && t - kRing < c.e)) {
          f2 dxv[P];
          bwd_dx<P>(g, gr, tap, dxv);
          if (STORE || active) store_row<VEC>(dxrow, dxv);
        }
      } else {
#pragma unroll
        for (int q = 0; q < P; ++q) g[q] = 0ull;  // rows before the range: only the x ring
      }
      rings_push<P>(h, gr, x, g);
    }
    dxrow += p.D;
  }
}

// Packed sequences: the dx formula's value at row u lands in dx (u in the sequence that
// starts at ss, inside [a, e)) or in the gradient of sequence i's initial state (u among the
// W-1 rows before ss, when this range holds the sequence's first row).
template <int VEC>
__device__ __forceinline__ void bwd_put(int u, int i, int ss, int se, const TileCursor& c,
                                        bool active, const BwdArgs& p, int64_t d0,
                                        const f2 (&v)[VEC / 2]) {
  if (!active) return;
  if (u >= ss && u >= c.a && u < c.e) {
    store_row<VEC>(p.dx + static_cast<int64_t>(u) * p.D + d0, v);
  } else if (p.dinit && i >= 0 && u < ss && u >= ss - (p.W - 1) && ss >= c.a && ss < c.e &&
             ss < se) {
    store_dinit<VEC>(p.dinit, i, p.D, p.W, u - (ss - (p.W - 1)), d0, v);
  }
}

// Packed sequences: the event at row t, where the current sequence ends and the next
// non-empty one starts.  The ending sequence's last W-1 dx rows (or, for a short sequence,
// its last initial-state gradient rows) are finished with g = 0 past its end; then both
// rings restart: x from the new sequence's initial state (fetched one sequence ahead), g
// from zeros.
template <int VEC>
__device__ __forceinline__ void bwd_boundary(int t, const TileCursor& c, SeqTracker& sq,
                                             bool active, const BwdArgs& p, int64_t d0,
                                             const f2 (&tap)[4][VEC / 2], f2 (&h)[3][VEC / 2],
                                             f2 (&gr)[3][VEC / 2], uint32_t (&hin)[3][VEC / 2],
                                             int& hin_seq) {
  constexpr int P = VEC / 2;
  f2 zero[P];
#pragma unroll
  for (int q = 0; q < P; ++q) zero[q] = 0ull;
#pragma unroll
  for (int m = 0; m < kRing; ++m) {
    f2 v[P];
    bwd_dx<P>(zero, gr, tap, v);
    bwd_put<VEC>(t - kRing + m, sq.i, sq.ss, t, c, active, p, d0, v);
#pragma unroll
    for (int q = 0; q < P; ++q) {
      gr[2][q] = gr[1][q];
      gr[1][q] = gr[0][q];
      gr[0][q] = 0ull;
    }
  }
  sq.next(t);
  if (hin_seq != sq.i) init_ring<VEC>(p.init, init_slot(p, sq.i), p.D, p.W, d0, active, hin);
  ring_of<VEC>(hin, p.W, h);
#pragma unroll
  for (int q = 0; q < P; ++q)
#pragma unroll
    for (int j = 0; j < 3; ++j) gr[j][q] = 0ull;
  hin_seq = -1;
  if (sq.i + 1 < p.nseq) {
    init_ring<VEC>(p.init, init_slot(p, sq.i + 1), p.D, p.W, d0, active, hin);
    hin_seq = sq.i + 1;
  }
}

// Packed sequences, a tile on the per-row path (the range's first and last tiles and tiles
// holding a sequence boundary or the rows just after one): rows before a fill the x ring,
// rows from a on give g (dw / dbias only inside [a, e)) and the dx value of row t - 3,
// which bwd_put files as dx or as initial-state gradient; a boundary event runs before the
// first row of each new sequence.  Halo rows past e finish the range's last dx rows.
template <int VEC, int R, bool ACT>
__device__ __forceinline__ void bwd_tile_vl(const uint8_t* xt, const uint8_t* dyt, int lane,
                                            const TileCursor& c, SeqTracker& sq, bool active,
                                            const BwdArgs& p, int64_t d0,
                                            const f2 (&tap)[4][VEC / 2],
                                            const f2 (&bias2)[VEC / 2], f2 (&h)[3][VEC / 2],
                                            f2 (&gr)[3][VEC / 2], f2 (&acc)[kRec][VEC / 2],
                                            uint32_t (&hin)[3][VEC / 2], int& hin_seq) {
  constexpr int P = VEC / 2;
  constexpr int ROWB = 32 * VEC * 2;
  // Not unrolled: unrolling the boundary event into every row made the whole kernel slower
  // (one sequence: 74.5 against 76.9 us), and running the rows between boundaries through an
  // unrolled loop with a row test was slower still with many sequences (128: 92.8 against
  // 87.1 us), measured.
#pragma unroll 1
  for (int i = 0; i < R; ++i) {
    const int t = c.tt + i;
    if (t >= c.from) {
      if (sq.at(t)) bwd_boundary<VEC>(t, c, sq, active, p, d0, tap, h, gr, hin, hin_seq);
      f2 x[P], g[P];
      smem_row<VEC>(xt + i * ROWB, lane, x);
      if (t >= c.a) {
        f2 dy[P];
        smem_row<VEC>(dyt + i * ROWB, lane, dy);
        bwd_g<P, ACT>(x, dy, h, tap, bias2, g);
        if (t < c.e) bwd_acc<P>(x, h, g, acc);
        f2 dxv[P];
        bwd_dx<P>(g, gr, tap, dxv);
        bwd_put<VEC>(t - kRing, sq.i, sq.ss, sq.nb, c, active, p, d0, dxv);
      } else {
#pragma unroll
        for (int q = 0; q < P; ++q) g[q] = 0ull;  // rows before the range: only the x ring
      }
      rings_push<P>(h, gr, x, g);
    }
  }
}

// Packed sequences: cu_seqlens into L2 before the dependency wait, so that the range search
// right after the wait, the first load the producer waits for, hits L2 instead of DRAM (the
// stream of the previous call has evicted it).  A prefetch returns no data and L2 is where
// device memory is coherent, so loads issued after the wait still see every write the
// previous kernel on the stream makes to cu_seqlens.  Measured at B*T = 16384, D = 4096:
// 72.1 -> 71.65 us per call for 16 mixed sequences, 69.8 -> 68.95 us for one.
__device__ __forceinline__ void prefetch_seqlens(const int32_t* cu, int nseq) {
  const int lines = (nseq + 32) / 32;  // entries 0 .. nseq, 32 per 128-byte line
  for (int k = 0; k < lines && k < 16; ++k)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(cu + 32 * k))
                 : "memory");
}

// Packed sequences, once per CTA: empty sequences get a zero initial-state gradient (CTA i,
// i + grid, ...), and CTA 0 checks cu_seqlens (a malformed one sets the fault word).  The
// `nthreads` threads from thread `first` on share the zeroing, and the warp holding thread
// `first` does the check; every call site runs it with whole warps.
__device__ __forceinline__ void bwd_varlen_once(const BwdArgs& p, int first, int nthreads) {
  const int tid = static_cast<int>(threadIdx.x) - first;
  const int lane = threadIdx.x & 31;
  if (p.dinit && p.W > 1) {
    const int64_t n = p.D * (p.W - 1);
    for (int i = blockIdx.x; i < p.nseq; i += gridDim.x) {
      if (clamp_row(p.cu[i + 1], p.BT) > clamp_row(p.cu[i], p.BT)) continue;
      uint16_t* o = p.dinit + static_cast<int64_t>(i) * n;
      for (int64_t k = tid; k < n; k += nthreads) o[k] = 0;
    }
  }
  if (blockIdx.x == 0 && tid < 32) {
    bool bad = false;
    for (int k = lane; k <= p.nseq; k += 32) {
      const int v = p.cu[k];
      if (v < 0 || v > p.BT || (k == 0 && v != 0) || (k == p.nseq && v != p.BT) ||
          (k > 0 && p.cu[k - 1] > v))
        bad = true;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&g_fault_bwd, kFaultSeqlens);
  }
}

// CTA: NW warps = SW neighbouring strips x RW = NW/SW consecutive row ranges (strips fastest,
// so at any time the CTA reads SW*32*VEC contiguous channels of the same rows); each warp
// runs its own TMA pipeline; the RW partial sums of each strip are added inside the CTA.
// MODE: kModeVarlen walks packed sequences (rows of [total, D], each sequence's ring from
// its initial state, its gradient written); kModeActNone leaves out the SiLU.
// The CTA's work is strip group sg (strips sg*SW .. sg*SW + SW - 1 of the problem) and range
// group rg; its partial-sum record slots are those of CTA blockIdx.x.
template <int VEC, int R, int S, int NW, int SW, int MODE>
__device__ __forceinline__ void bwd_cta(const CUtensorMap* tmx, const CUtensorMap* tmdy,
                                        const BwdArgs& p, int sg, int rg) {
  static_assert(NW % SW == 0, "SW strips must divide the CTA's warps");
  constexpr bool VL = (MODE & kModeVarlen) != 0;
  constexpr bool ACT = (MODE & kModeActNone) == 0;
  using Cursor = TileCursor;  // packed sequences: one batch row of T = total rows
  constexpr int RW = NW / SW;
  constexpr int CB = 32 * VEC;
  constexpr int P = VEC / 2;
  constexpr int TILE = R * CB * 2;
  constexpr int STAGE = 2 * TILE;  // x tile, then dy tile
  constexpr int REC = kRec * CB;   // floats in one partial record
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int si = warp % SW;
  const int cb = sg * SW + si;
  const int k = rg * RW + warp / SW;
  const bool has_work = cb < p.n_cb && k < p.wpc;

  uint8_t* stages = smem + warp * (S * STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * S * STAGE) + warp * S;

  const int c0 = cb * CB;
  const int64_t d0 = c0 + lane * VEC;
  const bool active = has_work && d0 < p.D;
  const bool all_active = c0 + CB <= p.D;  // uniform over the warp

  if (has_work && lane == 0) {
    prefetch_tensormap(tmx);
    prefetch_tensormap(tmdy);
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if constexpr (VL) prefetch_seqlens(p.cu, p.nseq);
  }
  __syncwarp();

  // Everything above reads no global memory (cu_seqlens is only prefetched into L2); from
  // here on the previous kernel on the stream has completed.
  grid_dependency_wait();
  grid_launch_dependents();  // the reduction waits for this grid in griddepcontrol.wait

  // The warp's row range, after the wait: packed sequences split it by cu_seqlens, which
  // the previous kernel on the stream may have written.
  int r0, r1;
  if constexpr (VL) {
    // Equal cost per range: a sequence boundary costs a warp the pulled-back last tile, the
    // halo, the ring refill and two tiles on the per-row path; 40-48 rows balanced 16 and
    // 128 mixed sequences and 8 short clustered ones best (measured).
    constexpr int kBoundaryRows = 44;
    cost_split_range(p.cu, p.nseq, p.BT, kBoundaryRows, k, p.wpc, lane, r0, r1);
  } else {
    r0 = static_cast<int>(static_cast<int64_t>(k) * p.BT / p.wpc);
    r1 = static_cast<int>(static_cast<int64_t>(k + 1) * p.BT / p.wpc);
  }

  f2 acc[kRec][P];
#pragma unroll
  for (int q = 0; q < P; ++q)
#pragma unroll
    for (int j = 0; j < kRec; ++j) acc[j][q] = 0ull;

  if (has_work) {
    Cursor pc, cc;
    pc.init(r0, r1, p.T, kRing, R);
    cc = pc;
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < S; ++s) {
        if (!pc.done) {
          mbar_arrive_expect_tx(&bars[s], STAGE);
          tma_load_3d(stages + s * STAGE, tmx, &bars[s], c0, pc.tt, pc.b, pol);
          tma_load_3d(stages + s * STAGE + TILE, tmdy, &bars[s], c0, pc.tt, pc.b, pol);
          pc.advance();
        }
      }
    }

    // Taps load while the first tiles are in flight.
    f2 tap[4][P], bias2[P];
    load_taps<VEC>(p.w, p.bias, p.wdt, p.W, d0, active, tap, bias2);

    f2 h[3][P], gr[3][P];
#pragma unroll
    for (int q = 0; q < P; ++q)
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        h[j][q] = 0ull;
        gr[j][q] = 0ull;
      }
    // Packed sequences: the sequence of the rows walked (from the first ring-fill row on),
    // and hin, the initial x ring of sequence hin_seq, fetched one sequence ahead.
    SeqTracker sq;
    uint32_t hin[3][P];
    int hin_seq = -1;
    if constexpr (VL) {
      sq.init(p.cu, p.nseq, p.BT, r0 - kRing, lane);  // all lanes of the warp
      if (sq.i + 1 < p.nseq) {
        init_ring<VEC>(p.init, init_slot(p, sq.i + 1), p.D, p.W, d0, active, hin);
        hin_seq = sq.i + 1;
      }
    }

    uint32_t parity = 0;
    int s = 0;
    while (!cc.done) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (parity >> s) & 1u,
                                                               kWaitLimitNs));
      if (!ok) {
        if (lane == 0) atomicOr(&g_fault_bwd, kFaultBwdWait);
        // Let this warp's other copies land (bounded) before its stages are reused.
        for (int j = 0; j < S; ++j)
          (void)mbar_wait_bounded(&bars[j], (parity >> j) & 1u, 100000000ull);
        break;
      }
      parity ^= 1u << s;
      const uint8_t* xt = stages + s * STAGE;
      bool full_tile = cc.from == cc.tt && cc.tt >= cc.a + kRing && cc.tt + R <= cc.e;
      if constexpr (VL)  // and no boundary inside, nor one within the 3 rows before
        full_tile = full_tile && cc.tt - kRing >= sq.ss &&
                    !(sq.i + 1 < p.nseq && sq.nb >= cc.tt && sq.nb < cc.tt + R);
      if (full_tile) {
        if (all_active)
          bwd_tile<VEC, R, true, true, ACT>(xt, xt + TILE, lane, cc, active, p, d0, tap, bias2, h, gr, acc);
        else
          bwd_tile<VEC, R, true, false, ACT>(xt, xt + TILE, lane, cc, active, p, d0, tap, bias2, h, gr, acc);
      } else if constexpr (VL) {
        bwd_tile_vl<VEC, R, ACT>(xt, xt + TILE, lane, cc, sq, active, p, d0, tap, bias2, h, gr,
                                 acc, hin, hin_seq);
      } else {
        bwd_tile<VEC, R, false, false, ACT>(xt, xt + TILE, lane, cc, active, p, d0, tap, bias2, h, gr, acc);
      }
      __syncwarp();
      if (lane == 0 && !pc.done) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[s], STAGE);
        tma_load_3d(stages + s * STAGE, tmx, &bars[s], c0, pc.tt, pc.b, pol);
        tma_load_3d(stages + s * STAGE + TILE, tmdy, &bars[s], c0, pc.tt, pc.b, pol);
        pc.advance();
      }
      cc.advance();
      s = (s + 1 == S) ? 0 : s + 1;
    }
  }
  if constexpr (VL) bwd_varlen_once(p, 0, NW * 32);

  // ---- the CTA's partial sums, added in a fixed order ------------------------------------
  // Every warp has consumed all its tiles, so the stage memory is free for NW records.
  __syncthreads();
  float* buf = reinterpret_cast<float*>(smem);  // [NW][kRec][CB], sums of g2 = 2g halved
#pragma unroll
  for (int j = 0; j < kRec; ++j) {
    float v[VEC];
#pragma unroll
    for (int q = 0; q < P; ++q) f2_unpack(f2_mul(acc[j][q], f2_splat(0.5f)), v[2 * q], v[2 * q + 1]);
#pragma unroll
    for (int q = 0; q < VEC; ++q) buf[warp * REC + j * CB + lane * VEC + q] = v[q];
  }
  __syncthreads();
  // Record slot si of this CTA: strip sg*SW + si summed over its RW ranges in range order.
  float* rec = p.ws + static_cast<int64_t>(blockIdx.x) * SW * REC;
  for (int e = threadIdx.x; e < SW * REC; e += NW * 32) {
    const int slot = e / REC;
    const int jc = e - slot * REC;
    float a = 0.f;
#pragma unroll
    for (int r = 0; r < RW; ++r) a += buf[(r * SW + slot) * REC + jc];
    rec[e] = a;
  }
}

template <int VEC, int R, int S, int NW, int SW, int MODE>
__global__ void __launch_bounds__(NW * 32, 1)
    cconv_bwd_kernel(const __grid_constant__ CUtensorMap tmx,
                     const __grid_constant__ CUtensorMap tmdy, const BwdArgs p) {
  const int n_sg = (p.n_cb + SW - 1) / SW;  // strip groups
  bwd_cta<VEC, R, S, NW, SW, MODE>(&tmx, &tmdy, p, blockIdx.x % n_sg, blockIdx.x / n_sg);
}

// Lockstep form of the backward: NC consumer warps own the NC neighbouring channel strips
// of one row range, and a producer warp (index NC) loads each stage's NC x tiles and NC dy
// tiles together, so a stage is R rows of NC*CB contiguous channels of both tensors.  A
// stage is re-armed once every consumer has released it (full / empty mbarriers).  Each
// consumer runs the same per-warp tile code as the independent-pipeline form (for packed
// sequences, with its own sequence tracking); the partial records have the same layout
// (SW = NC strips, one range per CTA).
template <int VEC, int R, int S, int NC, int MODE>
__device__ __forceinline__ void bwd_cta_ls(const CUtensorMap* tmx, const CUtensorMap* tmdy,
                                           const BwdArgs& p, int sg, int rg) {
  constexpr bool VL = (MODE & kModeVarlen) != 0;
  constexpr bool ACT = (MODE & kModeActNone) == 0;
  constexpr int CB = 32 * VEC;
  constexpr int P = VEC / 2;
  constexpr int TILE = R * CB * 2;
  constexpr int STAGE = 2 * NC * TILE;  // NC x tiles, then NC dy tiles
  constexpr int REC = kRec * CB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c0 = sg * NC * CB;
  int nact = static_cast<int>((p.D - c0 + CB - 1) / CB);  // consumer warps with channels
  if (nact > NC) nact = NC;

  if (threadIdx.x == 0) {
    prefetch_tensormap(tmx);
    prefetch_tensormap(tmdy);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nact);
    }
    fence_mbar_init();
    if constexpr (VL) prefetch_seqlens(p.cu, p.nseq);
  }
  __syncthreads();
  grid_dependency_wait();
  // The reduction launched after this kernel waits for its completion in
  // griddepcontrol.wait, so it may be scheduled now: its CTAs then sit resident and start
  // the moment this grid finishes (0.7 us per call at B=2 T=8192 D=4096, measured).
  grid_launch_dependents();

  // The row range, after the wait: packed sequences split it by cu_seqlens, which the
  // previous kernel on the stream may have written.
  int r0, r1;
  if constexpr (VL) {
    // Equal cost per range, a sequence boundary counting as kBoundaryRows rows.  Measured over
    // 16384 x 4096 rows with initial states, summed over ten length mixes of 8 to 128
    // sequences: 12 rows 750.0, 16: 734.9, 20: 734.9, 32: 740.6 us (16 and 32 alike at 16
    // sequences, 16 faster by 1.5 to 3.5 us at 64 and 128).  Before the initial rings stopped
    // stalling the warps at each boundary, 32 had measured best.
    constexpr int kBoundaryRows = 16;
    cost_split_range(p.cu, p.nseq, p.BT, kBoundaryRows, rg, p.wpc, lane, r0, r1);
  } else {
    r0 = static_cast<int>(static_cast<int64_t>(rg) * p.BT / p.wpc);
    r1 = static_cast<int>(static_cast<int64_t>(rg + 1) * p.BT / p.wpc);
  }

  f2 acc[kRec][P];
#pragma unroll
  for (int q = 0; q < P; ++q)
#pragma unroll
    for (int j = 0; j < kRec; ++j) acc[j][q] = 0ull;

  TileCursor cur;  // packed sequences: one batch row of T = total rows
  cur.init(r0, r1, p.T, kRing, R);
  if (warp == NC) {
    // ---- producer warp -------------------------------------------------------------------
    if (lane == 0) {
      uint32_t eph = 0;
      int s = 0, i = 0;
      for (; !cur.done; ++i) {
        if (i >= S) {  // wait until every consumer has released this stage
          if (!mbar_wait_bounded(&empty[s], (eph >> s) & 1u, kWaitLimitNs)) {
            atomicOr(&g_fault_bwd, kFaultBwdWait);
            break;
          }
          eph ^= 1u << s;
        }
        uint8_t* st = smem + s * STAGE;
        mbar_arrive_expect_tx(&full[s], 2 * nact * TILE);
        for (int w = 0; w < nact; ++w)
          tma_load_3d(st + w * TILE, tmx, &full[s], c0 + w * CB, cur.tt, cur.b);
        for (int w = 0; w < nact; ++w)
          tma_load_3d(st + (NC + w) * TILE, tmdy, &full[s], c0 + w * CB, cur.tt, cur.b);
        cur.advance();
        s = (s + 1 == S) ? 0 : s + 1;
      }
      drain_issued<S>(full, i);  // i stages issued
    }
  } else if (warp < nact) {
    // ---- consumer ------------------------------------------------------------------------
    const int64_t d0 = c0 + warp * CB + lane * VEC;
    const bool active = d0 < p.D;
    const bool all_active = c0 + nact * CB <= p.D && nact == NC;  // uniform over the CTA
    f2 tap[4][P], bias2[P];
    load_taps<VEC>(p.w, p.bias, p.wdt, p.W, d0, active, tap, bias2);
    f2 h[3][P], gr[3][P];
#pragma unroll
    for (int q = 0; q < P; ++q)
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        h[j][q] = 0ull;
        gr[j][q] = 0ull;
      }
    // Packed sequences: the sequence of the rows walked (from the first ring-fill row on),
    // and hin, the initial x ring of sequence hin_seq, fetched one sequence ahead.
    SeqTracker sq;
    uint32_t hin[3][P];
    int hin_seq = -1;
    if constexpr (VL) {
      sq.init(p.cu, p.nseq, p.BT, r0 - kRing, lane);  // all lanes of the warp
      if (sq.i + 1 < p.nseq) {
        init_ring<VEC>(p.init, init_slot(p, sq.i + 1), p.D, p.W, d0, active, hin);
        hin_seq = sq.i + 1;
      }
      // While the first stage is on its way: the check of cu_seqlens (in L2 by now) and the
      // zero gradients of empty sequences, which at the end held up the CTA's finish.
      bwd_varlen_once(p, 0, nact * 32);
    }
    uint32_t fph = 0;
    int s = 0;
    while (!cur.done) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (fph >> s) & 1u,
                                                               kWaitLimitNs));
      if (!ok) {
        if (lane == 0) atomicOr(&g_fault_bwd, kFaultBwdWait);
        // Let the copies already issued land (bounded) before the stages are reused.
        for (int j = 0; j < S; ++j)
          (void)mbar_wait_bounded(&full[j], (fph >> j) & 1u, 100000000ull);
        break;
      }
      fph ^= 1u << s;
      const uint8_t* xt = smem + s * STAGE + warp * TILE;
      const uint8_t* dyt = xt + NC * TILE;
      bool full_tile = cur.from == cur.tt && cur.tt >= cur.a + kRing && cur.tt + R <= cur.e;
      if constexpr (VL)  // and no boundary inside, nor one within the 3 rows before
        full_tile = full_tile && cur.tt - kRing >= sq.ss &&
                    !(sq.i + 1 < p.nseq && sq.nb >= cur.tt && sq.nb < cur.tt + R);
      if (full_tile) {
        if (all_active)
          bwd_tile<VEC, R, true, true, ACT>(xt, dyt, lane, cur, active, p, d0, tap, bias2, h, gr, acc);
        else
          bwd_tile<VEC, R, true, false, ACT>(xt, dyt, lane, cur, active, p, d0, tap, bias2, h, gr, acc);
      } else if constexpr (VL) {
        bwd_tile_vl<VEC, R, ACT>(xt, dyt, lane, cur, sq, active, p, d0, tap, bias2, h, gr, acc,
                                 hin, hin_seq);
      } else {
        bwd_tile<VEC, R, false, false, ACT>(xt, dyt, lane, cur, active, p, d0, tap, bias2, h, gr, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      cur.advance();
      s = (s + 1 == S) ? 0 : s + 1;
    }
  }

  // ---- the CTA's partial sums: one record per strip (one range per CTA) -------------------
  float* rec = p.ws + static_cast<int64_t>(blockIdx.x) * NC * REC;
  if (warp < NC) {
#pragma unroll
    for (int j = 0; j < kRec; ++j) {
      float v[VEC];
#pragma unroll
      for (int q = 0; q < P; ++q)
        f2_unpack(f2_mul(acc[j][q], f2_splat(0.5f)), v[2 * q], v[2 * q + 1]);
      float* o = rec + warp * REC + j * CB + lane * VEC;
      if constexpr (VEC == 4) {
        // 16-byte aligned: every workspace is (the host checks it; the no-alloc array is
        // 256-byte aligned), and each offset is a multiple of 4 floats.
        *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int q = 0; q < VEC; ++q) o[q] = v[q];
      }
    }
  }
}

template <int VEC, int R, int S, int NC, int MINB, int MODE>
__global__ void __launch_bounds__((NC + 1) * 32, MINB)
    cconv_bwd_ls_kernel(const __grid_constant__ CUtensorMap tmx,
                        const __grid_constant__ CUtensorMap tmdy, const BwdArgs p) {
  const int n_sg = (p.n_cb + NC - 1) / NC;
  bwd_cta_ls<VEC, R, S, NC, MODE>(&tmx, &tmdy, p, blockIdx.x % n_sg, blockIdx.x / n_sg);
}

// ------------------------------------------------------------------------------------
// Several problems in one launch (the q, k and v convolutions of a layer): the same rows
// and width, each its own x, dy, weights, outputs and D.  Each problem's strips are grouped
// SW at a time on their own (no CTA straddles two problems); CTA -> (strip group over all
// problems, range group), so every problem's records sit in one workspace.
// ------------------------------------------------------------------------------------
constexpr int kMaxProblems = 4;

struct BwdMulti {
  CUtensorMap mx[kMaxProblems];
  CUtensorMap mdy[kMaxProblems];
  BwdArgs base;                      // shared: ws, T, BT, wpc, W, wdt
  const void* w[kMaxProblems];
  const void* bias[kMaxProblems];
  uint16_t* dx[kMaxProblems];
  int64_t D[kMaxProblems];
  int n_cb[kMaxProblems];
  int sg0[kMaxProblems + 1];         // first strip group of each problem
  int n;
};

template <int VEC, int R, int S, int NW, int SW>
__global__ void __launch_bounds__(NW * 32, 1)
    cconv_bwd_multi_kernel(const __grid_constant__ BwdMulti m) {
  const int n_sg = m.sg0[m.n];
  const int sga = blockIdx.x % n_sg;
  int k = 0;
#pragma unroll
  for (int j = 1; j < kMaxProblems; ++j)
    if (j < m.n && sga >= m.sg0[j]) k = j;
  BwdArgs q = m.base;
  q.w = m.w[k];
  q.bias = m.bias[k];
  q.dx = m.dx[k];
  q.D = m.D[k];
  q.n_cb = m.n_cb[k];
  bwd_cta<VEC, R, S, NW, SW, 0>(&m.mx[k], &m.mdy[k], q, sga - m.sg0[k], blockIdx.x / n_sg);
}

// The same in the lockstep form (strip groups of NC strips per problem, one range per CTA).
template <int VEC, int R, int S, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 1)
    cconv_bwd_ls_multi_kernel(const __grid_constant__ BwdMulti m) {
  const int n_sg = m.sg0[m.n];
  const int sga = blockIdx.x % n_sg;
  int k = 0;
#pragma unroll
  for (int j = 1; j < kMaxProblems; ++j)
    if (j < m.n && sga >= m.sg0[j]) k = j;
  BwdArgs q = m.base;
  q.w = m.w[k];
  q.bias = m.bias[k];
  q.dx = m.dx[k];
  q.D = m.D[k];
  q.n_cb = m.n_cb[k];
  bwd_cta_ls<VEC, R, S, NC, 0>(&m.mx[k], &m.mdy[k], q, sga - m.sg0[k], blockIdx.x / n_sg);
}

// dw[d, W-1-lag] and dbias[d]: strip cb's records are slot cb % SW of the CTAs of strip group
// cb / SW (plus the problem's first strip group), one per range group.  CTA = 32 channels x
// kRedGroups groups for one record row j (blockIdx.y): group g adds range groups g, g + G,
// g + 2G, ... and the G group sums are then added in group order.  Deterministic; no
// atomics; a few independent loads per thread.  blockIdx.x runs over the 32-channel blocks
// of every problem in turn.
constexpr int kRedGroups = 8;

// One problem: the same sum with scalar arguments.
__global__ void __launch_bounds__(32 * kRedGroups)
    cconv_bwd_reduce1_kernel(const float* __restrict__ ws, int cb_width, int sw, int n_sg,
                             int n_rg, int64_t D, int W, int wdt, void* dw, void* dbias) {
  __shared__ float part[kRedGroups][33];
  grid_dependency_wait();
  grid_launch_dependents();  // the next kernel waits for this grid in griddepcontrol.wait
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x >> 5;
  const int j = blockIdx.y;
  // D < 2^31, so the channel index fits 32 bits; the CTA's 32 channels share one strip.
  const int d = static_cast<int>(blockIdx.x) * 32 + lane;
  float a = 0.f;
  if (d < D) {
    const int cb = static_cast<int>(blockIdx.x) / (cb_width / 32);
    const int c = d - cb * cb_width;
    const int64_t rec = static_cast<int64_t>(kRec) * cb_width;
    // strip cb is record cb % sw of strip group cb / sw: offset (sg * sw + si) * rec = cb * rec
    const float* base = ws + cb * rec + static_cast<int64_t>(j) * cb_width + c;
    const int64_t step = static_cast<int64_t>(n_sg) * sw * rec;  // next range group's CTA
    float a0 = 0.f, a1 = 0.f;
    int r = grp;
    for (; r + kRedGroups < n_rg; r += 2 * kRedGroups) {
      a0 += base[r * step];
      a1 += base[(r + kRedGroups) * step];
    }
    if (r < n_rg) a0 += base[r * step];
    a = a0 + a1;
  }
  part[grp][lane] = a;
  __syncthreads();
  if (grp != 0 || d >= D) return;
  float t = 0.f;
#pragma unroll
  for (int g = 0; g < kRedGroups; ++g) t += part[g][lane];
  if (j < 4) {
    const int lag = j;
    if (lag < W) {
      const int64_t o = static_cast<int64_t>(d) * W + (W - 1 - lag);
      if (wdt == CCONV_F32)
        static_cast<float*>(dw)[o] = t;
      else
        static_cast<uint16_t*>(dw)[o] = f32_to_bf16(t);
    }
  } else if (dbias) {
    if (wdt == CCONV_F32)
      static_cast<float*>(dbias)[d] = t;
    else
      static_cast<uint16_t*>(dbias)[d] = f32_to_bf16(t);
  }
}

struct RedArgs {
  const float* ws;
  int cb_width, sw, n_sg, n_rg;      // n_sg: strip groups of all problems
  int W, wdt, n;
  void* dw[kMaxProblems];
  void* dbias[kMaxProblems];
  int64_t D[kMaxProblems];
  int sg0[kMaxProblems];
  int blk0[kMaxProblems + 1];        // first 32-channel block of each problem
};

__global__ void __launch_bounds__(32 * kRedGroups) cconv_bwd_reduce_kernel(const RedArgs r) {
  __shared__ float part[kRedGroups][33];
  grid_dependency_wait();
  grid_launch_dependents();  // the next kernel waits for this grid in griddepcontrol.wait
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x >> 5;
  const int j = blockIdx.y;
  int k = 0;
#pragma unroll
  for (int u = 1; u < kMaxProblems; ++u)
    if (u < r.n && static_cast<int>(blockIdx.x) >= r.blk0[u]) k = u;
  const int64_t D = r.D[k];
  const int blk = static_cast<int>(blockIdx.x) - r.blk0[k];  // block within problem k
  const int d = blk * 32 + lane;                              // D < 2^31
  float a = 0.f;
  if (d < D) {
    const int cb = blk / (r.cb_width / 32);  // the CTA's 32 channels share one strip
    const int c = d - cb * r.cb_width;
    const int64_t rec = static_cast<int64_t>(kRec) * r.cb_width;
    // strip cb is record cb % sw of strip group sg0 + cb / sw: offset (sg0 * sw + cb) * rec
    const float* base = r.ws + (static_cast<int64_t>(r.sg0[k]) * r.sw + cb) * rec +
                        static_cast<int64_t>(j) * r.cb_width + c;
    const int64_t step = static_cast<int64_t>(r.n_sg) * r.sw * rec;  // next range group's CTA
    float a0 = 0.f, a1 = 0.f;
    int q = grp;
    for (; q + kRedGroups < r.n_rg; q += 2 * kRedGroups) {
      a0 += base[q * step];
      a1 += base[(q + kRedGroups) * step];
    }
    if (q < r.n_rg) a0 += base[q * step];
    a = a0 + a1;
  }
  part[grp][lane] = a;
  __syncthreads();
  if (grp != 0 || d >= D) return;
  float t = 0.f;
#pragma unroll
  for (int g = 0; g < kRedGroups; ++g) t += part[g][lane];
  const int W = r.W;
  if (j < 4) {
    const int lag = j;
    if (lag < W) {
      const int64_t o = static_cast<int64_t>(d) * W + (W - 1 - lag);
      if (r.wdt == CCONV_F32)
        static_cast<float*>(r.dw[k])[o] = t;
      else
        static_cast<uint16_t*>(r.dw[k])[o] = f32_to_bf16(t);
    }
  } else if (r.dbias[k]) {
    if (r.wdt == CCONV_F32)
      static_cast<float*>(r.dbias[k])[d] = t;
    else
      static_cast<uint16_t*>(r.dbias[k])[d] = f32_to_bf16(t);
  }
}

// One problem's reduction arguments.
static RedArgs red_args_one(const float* ws, int cb_width, int sw, int n_sg, int n_rg, int64_t D,
                            int W, int wdt, void* dw, void* dbias) {
  RedArgs r{};
  r.ws = ws;
  r.cb_width = cb_width;
  r.sw = sw;
  r.n_sg = n_sg;
  r.n_rg = n_rg;
  r.W = W;
  r.wdt = wdt;
  r.n = 1;
  r.dw[0] = dw;
  r.dbias[0] = dbias;
  r.D[0] = D;
  r.sg0[0] = 0;
  r.blk0[0] = 0;
  r.blk0[1] = static_cast<int>((D + 31) / 32);
  return r;
}

struct BwdConfig {
  int vec, rows, stages, warps, sw;
  int producer;  // 1: a producer warp beside the warps consumer warps (lockstep form)
  int minb;      // CTAs resident per SM
  void (*kernel)(const CUtensorMap, const CUtensorMap, const BwdArgs);
};

#define CCONV_BWD_CFG(V, R, S, NW, SW) \
  BwdConfig { V, R, S, NW, SW, 0, 1, cconv_bwd_kernel<V, R, S, NW, SW, 0> }
#define CCONV_BWD_LS_CFG(V, R, S, NC, M) \
  BwdConfig { V, R, S, NC, NC, 1, M, cconv_bwd_ls_kernel<V, R, S, NC, M, 0> }

// Entry 0 is the default from 2048 channels (16 strips of 128) up, entry 1 (4-strip
// lockstep CTAs) from 512 channels, and entry 2 (independent warp pipelines, 2-strip CTAs)
// below that.  Measured at B=2 T=8192 (us, entry 0 / 1 / 2):
//   D=512 17.7 / 16.9 / 17.1, 1024 27.2 / 24.4 / 25.2, 1536 39.7 / 33.4 / 34.3,
//   2048 40.3 / 40.5 / 40.3, 4096 66.9 / 74.5 / 72.2.
// Building with -DCCONV_TILE_SWEEP adds the other shapes that were measured against them,
// one of which the environment variable CCONV_BWD_CONFIG (an index into the table) then
// forces for every D; that build is for tile sweeps only, and its extra shapes are not
// covered by the parity tests.
static const BwdConfig kBwdConfigs[] = {
    CCONV_BWD_LS_CFG(4, 12, 4, 8, 1),
    CCONV_BWD_LS_CFG(4, 12, 6, 4, 1),
    CCONV_BWD_CFG(4, 12, 3, 8, 2),
#ifdef CCONV_TILE_SWEEP
    CCONV_BWD_CFG(4, 12, 3, 8, 4),
    CCONV_BWD_CFG(4, 12, 3, 8, 8),
    CCONV_BWD_CFG(4, 16, 3, 8, 4),
    CCONV_BWD_CFG(4, 12, 2, 12, 4),
    CCONV_BWD_LS_CFG(4, 16, 3, 8, 1),
    CCONV_BWD_LS_CFG(4, 12, 4, 4, 2),
    CCONV_BWD_LS_CFG(4, 12, 8, 4, 1),
#endif
};

static const BwdConfig& bwd_config(int64_t D) {
#ifdef CCONV_TILE_SWEEP
  static const int override_idx = [] {
    constexpr int n = sizeof(kBwdConfigs) / sizeof(kBwdConfigs[0]);
    const char* e = getenv("CCONV_BWD_CONFIG");
    const int v = e ? atoi(e) : -1;
    return (v >= 0 && v < n) ? v : -1;
  }();
  if (override_idx >= 0) return kBwdConfigs[override_idx];
#endif
  if (D >= 2048) return kBwdConfigs[0];
  return D >= 512 ? kBwdConfigs[1] : kBwdConfigs[2];
}

// Work split of the backward: strips of 32*VEC channels in groups of SW, each strip's rows in
// wpc ranges in groups of RW = warps/SW; one CTA per (strip group, range group).  wpc is a
// multiple of RW chosen so the grid is about one wave of the device's SMs.
struct BwdPlan {
  int n_cb, wpc, n_sg, n_rg, grid;
};

static int bwd_plan(int64_t B, int64_t T, int64_t D, const BwdConfig& cfg, BwdPlan* plan,
                    size_t* ws_bytes) {
  int sms = 0;
  const int rc = sm_count_current_device(&sms, nullptr);
  if (rc != CCONV_OK) return rc;
  const int rw = cfg.warps / cfg.sw;
  const int64_t cbw = 32 * cfg.vec;
  plan->n_cb = static_cast<int>((D + cbw - 1) / cbw);
  plan->n_sg = (plan->n_cb + cfg.sw - 1) / cfg.sw;
  int64_t n_rg = static_cast<int64_t>(sms) * cfg.minb / plan->n_sg;  // CTAs per strip group
  const int64_t by_rows = (B * T) / (32 * rw);           // ranges of at least 32 rows
  if (n_rg > by_rows) n_rg = by_rows;
  if (n_rg < 1) n_rg = 1;
  plan->n_rg = static_cast<int>(n_rg);
  plan->wpc = plan->n_rg * rw;
  plan->grid = plan->n_sg * plan->n_rg;
  *ws_bytes = static_cast<size_t>(plan->grid) * cfg.sw * kRec * cbw * sizeof(float);
  return CCONV_OK;
}

static int check_sizes(int64_t B, int64_t T, int64_t D, int W) {
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (B < 1 || T < 1 || D < 1 || B * T > (int64_t(1) << 31) - 16 || D > (int64_t(1) << 31) - 8)
    return CCONV_ERR_SHAPE;
  if (D % 8 != 0) return CCONV_ERR_ALIGN;
  return CCONV_OK;
}

}  // namespace cconv

extern "C" {

CCONV_API int cconv_bwd_workspace_bytes(int64_t B, int64_t T, int64_t D, int W, size_t* bytes) {
  using namespace cconv;
  if (!bytes) return CCONV_ERR_NULL;
  int rc = check_sizes(B, T, D, W);
  if (rc != CCONV_OK) return rc;
  BwdPlan plan;
  return bwd_plan(B, T, D, bwd_config(D), &plan, bytes);
}

CCONV_API int cconv_bwd(const void* x, int64_t sxb, int64_t sxt, const void* dy, int64_t sdb,
                        int64_t sdt, int64_t B, int64_t T, int64_t D, const void* w,
                        const void* bias, cconv_dtype wdt, int W, void* dx, void* dw,
                        void* dbias, void* workspace, size_t workspace_bytes,
                        cconv_stream_t stream) {
  using namespace cconv;
  if (!x || !dy || !w || !dx || !dw) return CCONV_ERR_NULL;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  int rc = check_sizes(B, T, D, W);
  if (rc != CCONV_OK) return rc;
  rc = check_rows_tensor(x, B, T, D, sxb, sxt);
  if (rc != CCONV_OK) return rc;
  rc = check_rows_tensor(dy, B, T, D, sdb, sdt);
  if (rc != CCONV_OK) return rc;
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(dx) % 16 != 0) return CCONV_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(w) % ew != 0 || reinterpret_cast<uintptr_t>(dw) % ew != 0)
    return CCONV_ERR_ALIGN;
  if ((bias && reinterpret_cast<uintptr_t>(bias) % ew != 0) ||
      (dbias && reinterpret_cast<uintptr_t>(dbias) % ew != 0))
    return CCONV_ERR_ALIGN;

  const BwdConfig& cfg = bwd_config(D);
  BwdPlan plan;
  size_t need = 0;
  rc = bwd_plan(B, T, D, cfg, &plan, &need);
  if (rc != CCONV_OK) return rc;
  if (!workspace || workspace_bytes < need) return CCONV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return CCONV_ERR_ALIGN;

  normalise_strides(B, T, D, sxb, sxt);
  normalise_strides(B, T, D, sdb, sdt);
  CUtensorMap tmx, tmdy;
  rc = encode_rows_map(&tmx, x, B, T, D, sxb, sxt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;
  rc = encode_rows_map(&tmdy, dy, B, T, D, sdb, sdt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;

  BwdArgs a{};
  a.w = w;
  a.bias = bias;
  a.dx = static_cast<uint16_t*>(dx);
  a.ws = static_cast<float*>(workspace);
  a.D = D;
  a.T = static_cast<int>(T);
  a.BT = static_cast<int>(B * T);
  a.n_cb = plan.n_cb;
  a.wpc = plan.wpc;
  a.W = W;
  a.wdt = wdt;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int smem = cfg.warps * cfg.stages * (2 * cfg.rows * 32 * cfg.vec * 2 + 8);
  const int red_bytes = cfg.warps * kRec * 32 * cfg.vec * static_cast<int>(sizeof(float));
  if (smem < red_bytes) smem = red_bytes;  // the stage memory doubles as the reduction buffer
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(cfg.kernel), smem);
  if (rc != CCONV_OK) return rc;
  if (launch_pdl(cfg.kernel, dim3(plan.grid), dim3((cfg.warps + cfg.producer) * 32), smem, st,
                 tmx, tmdy, a) !=
      cudaSuccess)
    return CCONV_ERR_CUDA;
  const float* wsp = a.ws;
  const int cbw = 32 * cfg.vec;
  const int sw = cfg.sw;
  const int n_sg = plan.n_sg;
  const int n_rg = plan.n_rg;
  const int wdt_i = static_cast<int>(wdt);
  if (launch_pdl(cconv_bwd_reduce1_kernel,
                 dim3(static_cast<unsigned>((D + 31) / 32), dbias ? kRec : W),
                 dim3(32 * kRedGroups), 0, st, wsp, cbw, sw, n_sg, n_rg, D, W, wdt_i, dw,
                 dbias) != cudaSuccess)
    return CCONV_ERR_CUDA;
  return CCONV_OK;
}

}  // extern "C"

namespace cconv {

// ------------------------------------------------------------------------------------
// cconv_bwd_noalloc: the backward with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they run the backward:
// an inference or training runtime that hands out memory only from an arena it sized up
// front, a plugin inside another framework that owns every allocation, or a host thread
// that must not call cudaMalloc because cudaMalloc can synchronise the device and stall
// other streams.  For them this entry point takes its per-warp partial sums from
// g_bwd_noalloc_scratch, a file-scope __device__ array of kBwdNoallocScratchBytes that every
// GPU loading this library holds until the process exits.  The caller still passes all
// inputs and outputs; nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// Host code cannot use the array's name as a device address (it names a host-side
// stand-in), so every call looks the address up with cudaGetSymbolAddress in the context
// current on the calling thread.  That lookup is cheap once the library's device code is
// loaded in the context; the first call in a context may load it, which reserves the array
// there and is not a stream operation, so make that first call before any stream capture
// (and before sizing a memory arena, which the array then no longer competes with).  No
// address is cached, so a device reset or another context current on the same device is
// safe.  All calls on a device share the array, which keeps whatever the last call left in
// it; nothing in it needs to start at zero, because every record is fully written before it
// is read.  Calls whose work overlaps on the GPU (for example on two streams) race on the
// array and must be serialised by the caller.
// ------------------------------------------------------------------------------------
constexpr size_t kBwdNoallocScratchBytes = size_t(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[kBwdNoallocScratchBytes];

static void* bwd_noalloc_scratch_address(int* status) {
  void* p = nullptr;
  if (report_cuda("cudaGetSymbolAddress", cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch)) !=
          cudaSuccess ||
      !p) {
    *status = CCONV_ERR_CUDA;
    return nullptr;
  }
  *status = CCONV_OK;
  return p;
}

}  // namespace cconv

extern "C" CCONV_API int cconv_bwd_noalloc(const void* x, int64_t sxb, int64_t sxt,
                                           const void* dy, int64_t sdb, int64_t sdt, int64_t B,
                                           int64_t T, int64_t D, const void* w,
                                           const void* bias, cconv_dtype wdt, int W, void* dx,
                                           void* dw, void* dbias, cconv_stream_t stream) {
  using namespace cconv;
  size_t need = 0;
  int rc = cconv_bwd_workspace_bytes(B, T, D, W, &need);
  if (rc != CCONV_OK) return rc;
  if (need > kBwdNoallocScratchBytes) return CCONV_ERR_WORKSPACE;  // too large for the array
  void* scratch = bwd_noalloc_scratch_address(&rc);
  if (rc != CCONV_OK) return rc;
  return cconv_bwd(x, sxb, sxt, dy, sdb, sdt, B, T, D, w, bias, wdt, W, dx, dw, dbias, scratch,
                   kBwdNoallocScratchBytes, stream);
}

namespace cconv {

// Packed sequences run 4-strip groups (two row ranges per CTA): with 2-strip groups a CTA
// holds four ranges, and the end-of-CTA sum waits for the one with the most sequence
// boundaries (128 sequences over 16384 x 4096: 121 us against 101 us, measured).
static void (*const kBwdVarlenKernels[2])(const CUtensorMap, const CUtensorMap, const BwdArgs) = {
    cconv_bwd_kernel<4, 12, 3, 8, 4, kModeVarlen>,
    cconv_bwd_kernel<4, 12, 3, 8, 4, kModeVarlen | kModeActNone>,
};
static const BwdConfig kBwdVarlenConfig = {4, 12, 3, 8, 4, 0, 1, nullptr};
// From 512 channels on, the lockstep forms (as for batched rows): 8 strips per CTA from
// 2048 channels, 4 below.
static void (*const kBwdVarlenLsKernels[2])(const CUtensorMap, const CUtensorMap, const BwdArgs) = {
    cconv_bwd_ls_kernel<4, 12, 4, 8, 1, kModeVarlen>,
    cconv_bwd_ls_kernel<4, 12, 4, 8, 1, kModeVarlen | kModeActNone>,
};
static void (*const kBwdVarlenLs4Kernels[2])(const CUtensorMap, const CUtensorMap, const BwdArgs) = {
    cconv_bwd_ls_kernel<4, 12, 6, 4, 1, kModeVarlen>,
    cconv_bwd_ls_kernel<4, 12, 6, 4, 1, kModeVarlen | kModeActNone>,
};
static const BwdConfig kBwdVarlenLsConfig = {4, 12, 4, 8, 8, 1, 1, nullptr};
static const BwdConfig kBwdVarlenLs4Config = {4, 12, 6, 4, 4, 1, 1, nullptr};

static const BwdConfig& varlen_config(int64_t D) {
  if (D >= 2048) return kBwdVarlenLsConfig;
  return D >= 512 ? kBwdVarlenLs4Config : kBwdVarlenConfig;
}

// Zeroes n bf16 values (the initial-state gradient when there are no rows at all).
__global__ void cconv_zero_u16_kernel(uint16_t* p, int64_t n) {
  grid_dependency_wait();
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[k] = 0;
  grid_launch_dependents();
}

static int check_varlen_sizes(int64_t total, int64_t D, int W, int64_t nseq) {
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (total < 0 || nseq < 1 || D < 1 || total > (int64_t(1) << 31) - 16 ||
      nseq > (int64_t(1) << 31) - 2 || D > (int64_t(1) << 31) - 8)
    return CCONV_ERR_SHAPE;
  if (D % 8 != 0) return CCONV_ERR_ALIGN;
  return CCONV_OK;
}

}  // namespace cconv

extern "C" {

CCONV_API int cconv_bwd_varlen_workspace_bytes(int64_t total, int64_t D, int W, size_t* bytes) {
  using namespace cconv;
  if (!bytes) return CCONV_ERR_NULL;
  int rc = check_varlen_sizes(total, D, W, 1);
  if (rc != CCONV_OK) return rc;
  BwdPlan plan;
  return bwd_plan(1, total, D, varlen_config(D), &plan, bytes);
}

CCONV_API int cconv_bwd_varlen(const void* x, int64_t sxt, const void* dy, int64_t sdt,
                               int64_t total, int64_t D, const int32_t* cu_seqlens, int64_t nseq,
                               const void* w, const void* bias, cconv_dtype wdt, int W,
                               cconv_activation act, const void* initial_state,
                               const int32_t* state_indices, int64_t S, int32_t* status_dev,
                               void* dx, void* dw, void* dbias, void* d_initial_state,
                               void* workspace, size_t workspace_bytes, cconv_stream_t stream) {
  using namespace cconv;
  if (!w || !dw || !cu_seqlens) return CCONV_ERR_NULL;
  if (total > 0 && (!x || !dy || !dx)) return CCONV_ERR_NULL;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  if (act != CCONV_ACT_SILU && act != CCONV_ACT_NONE) return CCONV_ERR_SHAPE;
  int rc = check_varlen_sizes(total, D, W, nseq);
  if (rc != CCONV_OK) return rc;
  if (reinterpret_cast<uintptr_t>(cu_seqlens) % 4 != 0) return CCONV_ERR_ALIGN;
  if (total > 0) {
    rc = check_rows_tensor(x, 1, total, D, 0, sxt);
    if (rc != CCONV_OK) return rc;
    rc = check_rows_tensor(dy, 1, total, D, 0, sdt);
    if (rc != CCONV_OK) return rc;
    if (reinterpret_cast<uintptr_t>(dx) % 16 != 0) return CCONV_ERR_ALIGN;
  }
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(w) % ew != 0 || reinterpret_cast<uintptr_t>(dw) % ew != 0)
    return CCONV_ERR_ALIGN;
  if ((bias && reinterpret_cast<uintptr_t>(bias) % ew != 0) ||
      (dbias && reinterpret_cast<uintptr_t>(dbias) % ew != 0))
    return CCONV_ERR_ALIGN;
  const int L = W - 1;
  if (L > 0 && ((initial_state && reinterpret_cast<uintptr_t>(initial_state) % 2 != 0) ||
                (d_initial_state && reinterpret_cast<uintptr_t>(d_initial_state) % 2 != 0)))
    return CCONV_ERR_ALIGN;
  if (state_indices) {
    if (!status_dev) return CCONV_ERR_NULL;
    if (S < 1 || S > CCONV_UPDATE_MAX_SLOTS) return CCONV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(state_indices) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(status_dev) % 4 != 0)
      return CCONV_ERR_ALIGN;
  }
  // With indices, one small kernel checks them (and writes the status words) after the
  // gradient kernels; unusable slots are read as zeros by the stream kernel meanwhile.
  auto check_indices = [&](cudaStream_t s) {
    return state_indices ? launch_index_check(state_indices, nseq, S, status_dev, s) : CCONV_OK;
  };

  const BwdConfig& cfg = varlen_config(D);
  BwdPlan plan;
  size_t need = 0;
  rc = bwd_plan(1, total, D, cfg, &plan, &need);
  if (rc != CCONV_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int wdt_i = static_cast<int>(wdt);
  const dim3 red_grid(static_cast<unsigned>((D + 31) / 32), dbias ? kRec : W);

  if (total == 0) {  // no rows: dw, dbias and the initial-state gradient are all zero
    if (L > 0 && d_initial_state) {
      const int64_t n = nseq * D * L;
      int64_t g = (n + 255) / 256;
      if (g > 1024) g = 1024;
      if (launch_pdl(cconv_zero_u16_kernel, dim3(static_cast<unsigned>(g)), dim3(256), 0, st,
                     static_cast<uint16_t*>(d_initial_state), n) != cudaSuccess)
        return CCONV_ERR_CUDA;
    }
    const RedArgs ra = red_args_one(nullptr, 32 * cfg.vec, cfg.sw, plan.n_sg, 0, D, W, wdt_i,
                                    dw, dbias);
    if (launch_pdl(cconv_bwd_reduce_kernel, red_grid, dim3(32 * kRedGroups), 0, st, ra) !=
        cudaSuccess)
      return CCONV_ERR_CUDA;
    return check_indices(st);
  }

  if (!workspace || workspace_bytes < need) return CCONV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return CCONV_ERR_ALIGN;
  int64_t sb = 0, sdb = 0;
  normalise_strides(1, total, D, sb, sxt);
  normalise_strides(1, total, D, sdb, sdt);
  CUtensorMap tmx, tmdy;
  rc = encode_rows_map(&tmx, x, 1, total, D, sb, sxt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;
  rc = encode_rows_map(&tmdy, dy, 1, total, D, sdb, sdt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;

  BwdArgs a{};
  a.w = w;
  a.bias = bias;
  a.dx = static_cast<uint16_t*>(dx);
  a.ws = static_cast<float*>(workspace);
  a.D = D;
  a.T = static_cast<int>(total);
  a.BT = static_cast<int>(total);
  a.n_cb = plan.n_cb;
  a.wpc = plan.wpc;
  a.W = W;
  a.wdt = wdt;
  a.cu = cu_seqlens;
  a.init = L > 0 ? static_cast<const uint16_t*>(initial_state) : nullptr;
  a.idx = state_indices;
  a.S = state_indices ? S : nseq;
  a.dinit = L > 0 ? static_cast<uint16_t*>(d_initial_state) : nullptr;
  a.nseq = static_cast<int>(nseq);

  auto kern = (!cfg.producer ? kBwdVarlenKernels
                : cfg.warps == 8 ? kBwdVarlenLsKernels
                                 : kBwdVarlenLs4Kernels)[act == CCONV_ACT_NONE ? 1 : 0];
  int smem = cfg.warps * cfg.stages * (2 * cfg.rows * 32 * cfg.vec * 2 + 8);
  const int red_bytes = cfg.warps * kRec * 32 * cfg.vec * static_cast<int>(sizeof(float));
  if (smem < red_bytes) smem = red_bytes;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (rc != CCONV_OK) return rc;
  if (launch_pdl(kern, dim3(plan.grid), dim3((cfg.warps + cfg.producer) * 32), smem, st, tmx,
                 tmdy, a) != cudaSuccess)
    return CCONV_ERR_CUDA;
  // One problem: the reduction with scalar arguments.  The table-driven kernel computes the
  // same sums in the same order, yet made the packed backward 0.6 us slower per call
  // (70.9 against 70.3 us at 16 sequences, B*T = 16384, D = 4096, measured).
  if (launch_pdl(cconv_bwd_reduce1_kernel, red_grid, dim3(32 * kRedGroups), 0, st,
                 static_cast<const float*>(a.ws), 32 * cfg.vec, cfg.sw, plan.n_sg, plan.n_rg, D,
                 W, wdt_i, dw, dbias) != cudaSuccess)
    return CCONV_ERR_CUDA;
  return check_indices(st);
}

}  // extern "C"

namespace cconv {

// Work split of the multi-problem backward (default tile shape): strip groups of every
// problem side by side, range groups sized so the grid is about one wave.
struct MultiPlan {
  int n_cb[kMaxProblems], sg0[kMaxProblems + 1];
  int n_rg, wpc, grid;
  size_t ws_bytes;
};

static const BwdConfig kBwdMultiConfig = {4, 12, 3, 8, 4, 0, 1, nullptr};
static const BwdConfig kBwdMultiLsConfig = {4, 12, 4, 8, 8, 1, 1, nullptr};
static const BwdConfig kBwdMultiLs4Config = {4, 12, 6, 4, 4, 1, 1, nullptr};

// The 8-strip lockstep form when every problem fills a group of 8 strips (D > 896) and
// there are at least two groups in all, as for the batched call from 2048 channels on; the
// 4-strip lockstep form when every problem fills a group of 4 (D > 384); else independent
// warp pipelines.
static const BwdConfig& multi_config(int n, const int64_t* D) {
  int64_t strips = 0, least = int64_t(1) << 62;
  for (int k = 0; k < n; ++k) {
    const int64_t c = (D[k] + 127) / 128;
    strips += c;
    if (c < least) least = c;
  }
  if (least >= 8 && strips >= 16) return kBwdMultiLsConfig;
  return least >= 4 ? kBwdMultiLs4Config : kBwdMultiConfig;
}

static int multi_plan(int n, const int64_t* D, int64_t B, int64_t T, MultiPlan* mp) {
  const BwdConfig& cfg = multi_config(n, D);
  int sms = 0;
  const int rc = sm_count_current_device(&sms, nullptr);
  if (rc != CCONV_OK) return rc;
  const int rw = cfg.warps / cfg.sw;
  const int64_t cbw = 32 * cfg.vec;
  int n_sg = 0;
  for (int k = 0; k < n; ++k) {
    mp->n_cb[k] = static_cast<int>((D[k] + cbw - 1) / cbw);
    mp->sg0[k] = n_sg;
    n_sg += (mp->n_cb[k] + cfg.sw - 1) / cfg.sw;
  }
  mp->sg0[n] = n_sg;
  int64_t n_rg = sms / n_sg;
  const int64_t by_rows = (B * T) / (32 * rw);
  if (n_rg > by_rows) n_rg = by_rows;
  if (n_rg < 1) n_rg = 1;
  mp->n_rg = static_cast<int>(n_rg);
  mp->wpc = mp->n_rg * rw;
  mp->grid = n_sg * mp->n_rg;
  mp->ws_bytes = static_cast<size_t>(mp->grid) * cfg.sw * kRec * cbw * sizeof(float);
  return CCONV_OK;
}

static int check_multi_sizes(int n, const int64_t* D, int64_t B, int64_t T, int W) {
  if (n < 1 || n > kMaxProblems) return CCONV_ERR_SHAPE;
  for (int k = 0; k < n; ++k) {
    const int rc = check_sizes(B, T, D[k], W);
    if (rc != CCONV_OK) return rc;
  }
  return CCONV_OK;
}

}  // namespace cconv

extern "C" {

CCONV_API int cconv_bwd_multi_workspace_bytes(int n, const int64_t* D, int64_t B, int64_t T,
                                              int W, size_t* bytes) {
  using namespace cconv;
  if (!bytes || !D) return CCONV_ERR_NULL;
  int rc = check_multi_sizes(n, D, B, T, W);
  if (rc != CCONV_OK) return rc;
  MultiPlan mp;
  rc = multi_plan(n, D, B, T, &mp);
  if (rc != CCONV_OK) return rc;
  *bytes = mp.ws_bytes;
  return CCONV_OK;
}

CCONV_API int cconv_bwd_multi(int n, const void* const* x, const int64_t* sxb,
                              const int64_t* sxt, const void* const* dy, const int64_t* sdb,
                              const int64_t* sdt, const int64_t* D, const void* const* w,
                              const void* const* bias, void* const* dx, void* const* dw,
                              void* const* dbias, int64_t B, int64_t T, cconv_dtype wdt, int W,
                              void* workspace, size_t workspace_bytes, cconv_stream_t stream) {
  using namespace cconv;
  if (!x || !sxb || !sxt || !dy || !sdb || !sdt || !D || !w || !dx || !dw) return CCONV_ERR_NULL;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  int rc = check_multi_sizes(n, D, B, T, W);
  if (rc != CCONV_OK) return rc;
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  bool any_dbias = false;
  for (int k = 0; k < n; ++k) {
    const void* bk = bias ? bias[k] : nullptr;
    void* dbk = dbias ? dbias[k] : nullptr;
    any_dbias = any_dbias || dbk;
    if (!x[k] || !dy[k] || !w[k] || !dx[k] || !dw[k]) return CCONV_ERR_NULL;
    rc = check_rows_tensor(x[k], B, T, D[k], sxb[k], sxt[k]);
    if (rc != CCONV_OK) return rc;
    rc = check_rows_tensor(dy[k], B, T, D[k], sdb[k], sdt[k]);
    if (rc != CCONV_OK) return rc;
    if (reinterpret_cast<uintptr_t>(dx[k]) % 16 != 0) return CCONV_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(w[k]) % ew != 0 || reinterpret_cast<uintptr_t>(dw[k]) % ew != 0)
      return CCONV_ERR_ALIGN;
    if ((bk && reinterpret_cast<uintptr_t>(bk) % ew != 0) ||
        (dbk && reinterpret_cast<uintptr_t>(dbk) % ew != 0))
      return CCONV_ERR_ALIGN;
  }
  MultiPlan mp;
  rc = multi_plan(n, D, B, T, &mp);
  if (rc != CCONV_OK) return rc;
  if (!workspace || workspace_bytes < mp.ws_bytes) return CCONV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return CCONV_ERR_ALIGN;

  const BwdConfig& cfg = multi_config(n, D);
  BwdMulti m;
  BwdArgs& a = m.base;
  a = BwdArgs{};
  a.ws = static_cast<float*>(workspace);
  a.T = static_cast<int>(T);
  a.BT = static_cast<int>(B * T);
  a.wpc = mp.wpc;
  a.W = W;
  a.wdt = wdt;
  RedArgs ra{};
  ra.ws = a.ws;
  ra.cb_width = 32 * cfg.vec;
  ra.sw = cfg.sw;
  ra.n_sg = mp.sg0[n];
  ra.n_rg = mp.n_rg;
  ra.W = W;
  ra.wdt = static_cast<int>(wdt);
  ra.n = n;
  int blk = 0;
  for (int k = 0; k < kMaxProblems; ++k) {
    const int src = k < n ? k : n - 1;  // unused slots: copies of the last problem
    int64_t sb = sxb[src], st = sxt[src], db = sdb[src], dt = sdt[src];
    normalise_strides(B, T, D[src], sb, st);
    normalise_strides(B, T, D[src], db, dt);
    rc = encode_rows_map(&m.mx[k], x[src], B, T, D[src], sb, st, 32 * cfg.vec, cfg.rows);
    if (rc != CCONV_OK) return rc;
    rc = encode_rows_map(&m.mdy[k], dy[src], B, T, D[src], db, dt, 32 * cfg.vec, cfg.rows);
    if (rc != CCONV_OK) return rc;
    m.w[k] = w[src];
    m.bias[k] = bias ? bias[src] : nullptr;
    m.dx[k] = static_cast<uint16_t*>(dx[src]);
    m.D[k] = D[src];
    m.n_cb[k] = mp.n_cb[src];
    m.sg0[k] = k < n ? mp.sg0[k] : mp.sg0[n];
    ra.dw[k] = dw[src];
    ra.dbias[k] = dbias ? dbias[src] : nullptr;
    ra.D[k] = D[src];
    ra.sg0[k] = mp.sg0[src];
    ra.blk0[k] = blk;
    if (k < n) blk += static_cast<int>((D[k] + 31) / 32);
  }
  m.sg0[kMaxProblems] = mp.sg0[n];
  ra.blk0[kMaxProblems] = blk;
  for (int k = n; k <= kMaxProblems; ++k) ra.blk0[k] = blk;
  m.n = n;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto kern = !cfg.producer   ? cconv_bwd_multi_kernel<4, 12, 3, 8, 4>
              : cfg.warps == 8 ? cconv_bwd_ls_multi_kernel<4, 12, 4, 8>
                               : cconv_bwd_ls_multi_kernel<4, 12, 6, 4>;
  int smem = cfg.warps * cfg.stages * (2 * cfg.rows * 32 * cfg.vec * 2 + 8);
  const int red_bytes = cfg.warps * kRec * 32 * cfg.vec * static_cast<int>(sizeof(float));
  if (smem < red_bytes) smem = red_bytes;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (rc != CCONV_OK) return rc;
  if (launch_pdl(kern, dim3(mp.grid), dim3((cfg.warps + cfg.producer) * 32), smem, st, m) !=
      cudaSuccess)
    return CCONV_ERR_CUDA;
  if (launch_pdl(cconv_bwd_reduce_kernel, dim3(static_cast<unsigned>(blk), any_dbias ? kRec : W),
                 dim3(32 * kRedGroups), 0, st, ra) != cudaSuccess)
    return CCONV_ERR_CUDA;
  return CCONV_OK;
}

}  // extern "C"
