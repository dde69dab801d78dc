// fwd.cu -- cconv_fwd and its packed-sequence and multi-problem forms: the forward stream.
//
// y[b,t,d] = silu(bias[d] + sum_{k<W} w[d,W-1-k] * x[b,t-k,d]), x = 0 left of the sequence.
// Definition: kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py (`_tap`,
// `_ld_ring`, `_silu`, `_fwd4`); its module docstring gives the design point this kernel
// keeps: one load of x, one sigmoid and one store per element, the W-1 previous rows held
// in registers.
//
// What differs from that Triton design: x does not travel through registers on its way in.
// Each CTA is warp-specialised: a producer warp keeps S stages of R rows x (NC*32*VEC)
// channels in flight into shared memory with TMA (one box per consumer warp, completing on
// the stage's "full" mbarrier), and NC consumer warps walk the stages in lockstep, each
// releasing a stage on its "empty" mbarrier.  Bytes in flight per SM are set by shared
// memory rather than by the register budget, which was the limit the pages measured, and the
// lockstep keeps the warps of an SM finishing together.  The 3 ring rows before a range and
// the zero padding before t = 0 come from the same tiled copy (out-of-range rows fill with
// zeros).  Arithmetic is packed f32x2; the sigmoid is 0.5 * tanh.approx(z/2) + 0.5.
//
// The same body also serves packed sequences (kModeVarlen: rows of [total, D], sequence
// boundaries as events at single rows, final states from the register ring, plus
// cconv_fwd_state_kernel for in-place or indexed states), no activation (kModeActNone), and
// several problems in one launch (cconv_fwd_multi_kernel).
#include <type_traits>

#include "strip.cuh"

namespace cconv {

static __device__ unsigned g_fault_fwd = 0;

int read_clear_fault_fwd(unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbol(out, g_fault_fwd, sizeof(unsigned)) != cudaSuccess) return CCONV_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_fault_fwd, &zero, sizeof(unsigned)) != cudaSuccess) return CCONV_ERR_CUDA;
  return CCONV_OK;
}

struct FwdArgs {
  const void* w;
  const void* bias;
  uint16_t* y;  // [B,T,D] contiguous bf16 ([total, D] for packed sequences)
  int64_t D;
  int T, BT;
  int cpc;      // CTAs per channel group
  int W, wdt;
  // packed sequences only
  const int32_t* cu;        // [nseq + 1] row offsets
  const uint16_t* init;     // [S, D, W-1] initial states, or null (zeros)
  const int32_t* idx;       // [nseq] slot of each sequence, or null (slot i)
  uint16_t* fin;            // [nseq, D, W-1] final states written by this kernel, or null
  int64_t S;
  int nseq;
};

// Kernel modes: the batched [B,T,D] form with SiLU is mode 0.
enum : int { kModeVarlen = 1, kModeActNone = 2 };

// One output row from the new input row x and the ring h = (x[t-1], x[t-2], x[t-3]).
// With halved taps hz = z / 2, and silu(z) = hz * (1 + tanh(hz)).
// Without the activation y = z = 2 hz.
template <int P, bool ACT>
__device__ __forceinline__ void fwd_row(const f2 (&x)[P], const f2 (&h)[3][P],
                                        const f2 (&tap)[4][P], const f2 (&bias2)[P],
                                        f2 (&yv)[P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    f2 hz = f2_fma(tap[0][q], x[q], bias2[q]);
    hz = f2_fma(tap[1][q], h[0][q], hz);
    hz = f2_fma(tap[2][q], h[1][q], hz);
    hz = f2_fma(tap[3][q], h[2][q], hz);
    yv[q] = ACT ? f2_fma(hz, f2_tanh(hz), hz) : f2_add(hz, hz);
  }
}

template <int P>
__device__ __forceinline__ void ring_push(f2 (&h)[3][P], const f2 (&x)[P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    h[2][q] = h[1][q];
    h[1][q] = h[0][q];
    h[0][q] = x[q];
  }
}

// Rows of one tile for this lane.  FULL: every row lies inside the segment.  Otherwise rows
// before `from` were done with the previous tile, rows before a only fill the ring, and rows
// from e on are not needed.  STORE: this lane's channels exist (every lane of a CTA whose
// channel group lies inside D), so stores need no per-row test.  The output row pointer
// advances by D per row.
template <int VEC, int R, bool FULL, bool STORE, bool ACT>
__device__ __forceinline__ void fwd_tile(const uint8_t* tile, int lane, const TileCursor& c,
                                         bool active, const FwdArgs& p, int64_t d0,
                                         const f2 (&tap)[4][VEC / 2], const f2 (&bias2)[VEC / 2],
                                         f2 (&h)[3][VEC / 2]) {
  constexpr int P = VEC / 2;
  constexpr int ROWB = 32 * VEC * 2;
  uint16_t* yrow = p.y + (static_cast<int64_t>(c.b) * p.T + c.tt) * p.D + d0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int t = c.tt + i;
    if (FULL || t >= c.from) {
      f2 x[P];
      smem_row<VEC>(tile + i * ROWB, lane, x);
      if (FULL || (t >= c.a && t < c.e)) {
        f2 yv[P];
        fwd_row<P, ACT>(x, h, tap, bias2, yv);
        if (STORE || active) store_row<VEC>(yrow, yv);
      }
      ring_push<P>(h, x);
    }
    yrow += p.D;
  }
}

// Loads one tile (rows cur.tt .. cur.tt+R-1, one box per consumer warp) into a stage.
template <int VEC, int R, int NC, class Cursor>
__device__ __forceinline__ void fwd_issue(uint8_t* st, uint64_t* full, const CUtensorMap* tmx,
                                          const Cursor& cur, int nact, int c0) {
  constexpr int CB = 32 * VEC;
  constexpr int TILE = R * CB * 2;
  mbar_arrive_expect_tx(full, nact * TILE);
  for (int w = 0; w < nact; ++w)
    tma_load_3d(st + w * TILE, tmx, full, c0 + w * CB, cur.tt, cur.b);
}

// Slot of sequence i in the state arrays, or -1 when the index is unusable (the state
// kernel reports it; here such a sequence just starts from zeros).
__device__ __forceinline__ int64_t seq_slot(const FwdArgs& p, int i) {
  const int64_t s = p.idx ? static_cast<int64_t>(p.idx[i]) : i;
  return (s >= 0 && s < p.S) ? s : -1;
}

// Packed sequences: checks cu_seqlens (cu[0] = 0, non-decreasing, cu[nseq] = total) with
// the 32 lanes of one warp, and raises the fault bit if it is ill-formed.
__device__ __forceinline__ void check_seqlens(const int32_t* cu, int nseq, int total, int lane,
                                              unsigned* fault) {
  bool bad = false;
  for (int k = lane; k <= nseq; k += 32) {
    const int v = cu[k];
    if (v < 0 || v > total || (k == 0 && v != 0) || (k == nseq && v != total) ||
        (k > 0 && cu[k - 1] > v))
      bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(fault, kFaultSeqlens);
}

// Final state of sequence i from the ring after its last row: entry j (row se - (W-1) + j)
// is h[W-2-j].  The ring holds exact bf16 values, so the conversion back is exact.
template <int VEC>
__device__ __forceinline__ void store_final(uint16_t* fin, int64_t i, int64_t D, int W,
                                            int64_t d0, const f2 (&h)[3][VEC / 2]) {
  const int L = W - 1;
  uint16_t* o = fin + (i * D + d0) * L;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (k >= L) break;
    const int j = L - 1 - k;
#pragma unroll
    for (int q = 0; q < VEC / 2; ++q) {
      float lo, hi;
      f2_unpack(h[k][q], lo, hi);
      o[(2 * q) * L + j] = f32_to_bf16(lo);
      o[(2 * q + 1) * L + j] = f32_to_bf16(hi);
    }
  }
}

// Final states of empty sequences (their initial state, or zeros) for sequences
// i = first, first + step, ...: one warp, 16-byte copies.
__device__ __forceinline__ void final_of_empty(const FwdArgs& p, int first, int step, int lane) {
  const int64_t n16 = p.D * (p.W - 1) / 8;  // uint4 per sequence
  for (int i = first; i < p.nseq; i += step) {
    if (clamp_row(p.cu[i + 1], p.BT) > clamp_row(p.cu[i], p.BT)) continue;
    uint4* o = reinterpret_cast<uint4*>(p.fin + static_cast<int64_t>(i) * p.D * (p.W - 1));
    const uint4* src = p.init ? reinterpret_cast<const uint4*>(
                                    p.init + static_cast<int64_t>(i) * p.D * (p.W - 1))
                              : nullptr;
    for (int64_t k = lane; k < n16; k += 32) o[k] = src ? src[k] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Packed sequences: the event at row t, where the current sequence ends and the next
// non-empty one starts.  The ending sequence's final state is its ring (if its last row is
// in this range); the ring then restarts from the new sequence's initial state, which was
// fetched one sequence ahead (hin); the one after it is fetched now.
template <int VEC>
__device__ __forceinline__ void fwd_boundary(int t, const TileCursor& c, SeqTracker& sq,
                                             bool active, const FwdArgs& p, int64_t d0,
                                             f2 (&h)[3][VEC / 2], uint32_t (&hin)[3][VEC / 2],
                                             int& hin_seq) {
  if (p.fin && active && sq.i >= 0 && sq.ss < t && t > c.a && t <= c.e)
    store_final<VEC>(p.fin, sq.i, p.D, p.W, d0, h);
  sq.next(t);
  if (hin_seq != sq.i) init_ring<VEC>(p.init, seq_slot(p, sq.i), p.D, p.W, d0, active, hin);
  ring_of<VEC>(hin, p.W, h);
  hin_seq = -1;
  if (sq.i + 1 < p.nseq) {
    init_ring<VEC>(p.init, seq_slot(p, sq.i + 1), p.D, p.W, d0, active, hin);
    hin_seq = sq.i + 1;
  }
}

// Packed sequences, a tile on the per-row path (the range's first and last tiles and tiles
// holding a sequence boundary): rows before a fill the ring, rows in [a, e) are computed,
// and a boundary event runs before the first row of each new sequence.  The ring stops at
// the range's last row, so after the loop it holds the final state of a sequence ending
// there.
template <int VEC, int R, bool ACT>
__device__ __forceinline__ void fwd_tile_vl(const uint8_t* tile, int lane, const TileCursor& c,
                                            SeqTracker& sq, bool active, const FwdArgs& p,
                                            int64_t d0, const f2 (&tap)[4][VEC / 2],
                                            const f2 (&bias2)[VEC / 2], f2 (&h)[3][VEC / 2],
                                            uint32_t (&hin)[3][VEC / 2], int& hin_seq) {
  constexpr int P = VEC / 2;
  constexpr int ROWB = 32 * VEC * 2;
  uint16_t* yrow = p.y + static_cast<int64_t>(c.tt) * p.D + d0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int t = c.tt + i;
    if (t >= c.from && t < c.e) {
      if (sq.at(t)) fwd_boundary<VEC>(t, c, sq, active, p, d0, h, hin, hin_seq);
      f2 x[P];
      smem_row<VEC>(tile + i * ROWB, lane, x);
      if (t >= c.a) {
        f2 yv[P];
        fwd_row<P, ACT>(x, h, tap, bias2, yv);
        if (active) store_row<VEC>(yrow, yv);
      }
      ring_push<P>(h, x);
    }
    yrow += p.D;
  }
}

// CTA: NC consumer warps (warp w owns channels c0 + w*CB .. c0 + (w+1)*CB - 1 of every tile).
// SEP: a separate producer warp (index NC) streams the stages; otherwise lane 0 of consumer
// warp 0 re-arms each stage once every consumer has released it.  Stage layout: NC boxes of
// R rows x CB channels.  MODE: kModeVarlen walks packed sequences (rows of [total, D], ring
// from each sequence's initial state); kModeActNone leaves out the SiLU.
//
// The CTA's work is channel group cg of the rows' range `part`; the kernels below pick them
// (and, for several problems in one launch, the problem) from blockIdx.x.
template <int VEC, int R, int S, int NC, bool SEP, int MODE>
__device__ __forceinline__ void fwd_cta(const CUtensorMap* tmx, const FwdArgs& p, int cg,
                                        int part) {
  // Cost of a sequence boundary in rows: the value that balanced the ranges best over
  // 16 and 128 mixed sequences and 8 short ones clustered together (16-24 measured alike).
  constexpr int kBoundaryRows = 20;
  constexpr bool VL = (MODE & kModeVarlen) != 0;
  constexpr bool ACT = (MODE & kModeActNone) == 0;
  static_assert(SEP || !VL, "packed sequences use the producer warp to check cu_seqlens");
  using Cursor = TileCursor;
  constexpr int CB = 32 * VEC;
  constexpr int TILE = R * CB * 2;
  constexpr int STAGE = NC * TILE;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c0 = cg * NC * CB;
  int nact = static_cast<int>((p.D - c0 + CB - 1) / CB);  // consumer warps with channels
  if (nact > NC) nact = NC;

  if (threadIdx.x == 0) {
    prefetch_tensormap(tmx);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nact);
    }
    fence_mbar_init();
  }
  __syncthreads();  // the only CTA-wide barrier

  // Nothing above touches global memory; from here on the previous kernel on the stream has
  // completed.
  grid_dependency_wait();
  // The next kernel waits for this whole grid in griddepcontrol.wait, so it may be
  // scheduled now and start the moment this grid finishes.
  grid_launch_dependents();

  // The row range, after the wait: packed sequences split it by cu_seqlens, which the
  // previous kernel on the stream may have written.
  int r0, r1;
  if constexpr (VL) {  // equal cost: a sequence boundary counts as kBoundaryRows rows
    cost_split_range(p.cu, p.nseq, p.BT, kBoundaryRows, part, p.cpc, lane, r0, r1);
  } else {
    r0 = static_cast<int>(static_cast<int64_t>(part) * p.BT / p.cpc);
    r1 = static_cast<int>(static_cast<int64_t>(part + 1) * p.BT / p.cpc);
  }
  Cursor cur;  // packed sequences: one batch row of T = total rows
  cur.init(r0, r1, p.T, 0, R);
  if (SEP && warp == NC) {
    // ---- producer warp -------------------------------------------------------------------
    int issued = 0;
    if (lane == 0) {
      uint32_t eph = 0;
      int s = 0, i = 0;
      for (; !cur.done; ++i) {
        if (i >= S) {  // wait until every consumer has released this stage
          if (!mbar_wait_bounded(&empty[s], (eph >> s) & 1u, kWaitLimitNs)) {
            atomicOr(&g_fault_fwd, kFaultFwdWait);
            break;
          }
          eph ^= 1u << s;
        }
        fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], tmx, cur, nact, c0);
        cur.advance();
        s = (s + 1 == S) ? 0 : s + 1;
      }
      issued = i;
    }
    if constexpr (VL) {  // the idle warp's packed-sequence duties overlap the last tiles
      __syncwarp();
      if (blockIdx.x == 0) check_seqlens(p.cu, p.nseq, p.BT, lane, &g_fault_fwd);
      if (p.fin) final_of_empty(p, blockIdx.x, gridDim.x, lane);
    }
    if (lane == 0) drain_issued<S>(full, issued);
  } else if (warp < nact) {
    // ---- consumer ------------------------------------------------------------------------
    const bool leader = !SEP && warp == 0;
    Cursor pc = cur;  // the leader's producer cursor, S tiles ahead
    int issued = 0;   // tiles the leader has issued
    if (leader && lane == 0) {
      for (int s = 0; s < S && !pc.done; ++s) {
        fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], tmx, pc, nact, c0);
        pc.advance();
        ++issued;
      }
    }
    const int64_t d0 = c0 + warp * CB + lane * VEC;
    const bool active = d0 < p.D;
    const bool all_active = c0 + NC * CB <= p.D;  // uniform over the CTA
    f2 tap[4][VEC / 2], bias2[VEC / 2];
    load_taps<VEC>(p.w, p.bias, p.wdt, p.W, d0, active, tap, bias2);
    f2 h[3][VEC / 2];
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
      for (int q = 0; q < VEC / 2; ++q) h[j][q] = 0ull;
    // Packed sequences: the sequence of the rows walked (from the first ring-fill row on),
    // and hin, the initial ring of sequence hin_seq, fetched one sequence ahead.
    SeqTracker sq;
    uint32_t hin[3][VEC / 2];
    int hin_seq = -1;
    if constexpr (VL) {
      sq.init(p.cu, p.nseq, p.BT, r0 - kRing, lane);  // all lanes of the warp
      if (sq.i + 1 < p.nseq) {
        init_ring<VEC>(p.init, seq_slot(p, sq.i + 1), p.D, p.W, d0, active, hin);
        hin_seq = sq.i + 1;
      }
    }

    uint32_t fph = 0, eph = 0;
    int s = 0;
    while (!cur.done) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (fph >> s) & 1u,
                                                               kWaitLimitNs));
      if (!ok) {
        if (lane == 0) atomicOr(&g_fault_fwd, kFaultFwdWait);
        break;
      }
      fph ^= 1u << s;
      const uint8_t* tile = smem + s * STAGE + warp * TILE;
      bool full_tile = cur.from == cur.tt && cur.tt >= cur.a && cur.tt + R <= cur.e;
      if constexpr (VL)  // and no sequence boundary inside
        full_tile = full_tile && !(sq.i + 1 < p.nseq && sq.nb >= cur.tt && sq.nb < cur.tt + R);
      if (full_tile) {
        if (all_active)
          fwd_tile<VEC, R, true, true, ACT>(tile, lane, cur, active, p, d0, tap, bias2, h);
        else
          fwd_tile<VEC, R, true, false, ACT>(tile, lane, cur, active, p, d0, tap, bias2, h);
      } else if constexpr (VL) {
        fwd_tile_vl<VEC, R, ACT>(tile, lane, cur, sq, active, p, d0, tap, bias2, h, hin, hin_seq);
      } else {
        fwd_tile<VEC, R, false, false, ACT>(tile, lane, cur, active, p, d0, tap, bias2, h);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (leader) {
        // Re-arm this stage with the tile S ahead once every consumer has released it.
        bool fine = true;
        if (lane == 0 && !pc.done) {
          fine = mbar_wait_bounded(&empty[s], (eph >> s) & 1u, kWaitLimitNs);
          if (fine) {
            fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], tmx, pc, nact, c0);
            pc.advance();
            ++issued;
          } else {
            atomicOr(&g_fault_fwd, kFaultFwdWait);
          }
        }
        eph ^= 1u << s;
        if (!__all_sync(0xffffffffu, fine)) break;
      }
      cur.advance();
      s = (s + 1 == S) ? 0 : s + 1;
    }
    if (leader && lane == 0) drain_issued<S>(full, issued);
    if constexpr (VL) {  // a sequence that ends exactly at the range's end
      if (p.fin && active && sq.i >= 0 && sq.nb == r1 && sq.ss < r1 && r0 < r1)
        store_final<VEC>(p.fin, sq.i, p.D, p.W, d0, h);
    }
  }
}

template <int VEC, int R, int S, int NC, int MINB, bool SEP, int MODE>
__global__ void __maxnreg__(regs_for(NC + SEP, MINB))
cconv_fwd_kernel(const __grid_constant__ CUtensorMap tmx, const FwdArgs p) {
  const int cg = blockIdx.x / p.cpc;
  fwd_cta<VEC, R, S, NC, SEP, MODE>(&tmx, p, cg, blockIdx.x - cg * p.cpc);
}

// ------------------------------------------------------------------------------------
// Several problems in one launch (the q, k and v convolutions of a layer): the same rows
// (B, T) and width, each its own x, weights, output and D.  The grid is every problem's
// channel groups x cpc row ranges; CTA -> (problem, channel group, range).
// ------------------------------------------------------------------------------------
constexpr int kMaxProblems = 4;

struct FwdMulti {
  CUtensorMap map[kMaxProblems];
  FwdArgs base;                      // shared: T, BT, cpc, W, wdt
  const void* w[kMaxProblems];
  const void* bias[kMaxProblems];
  uint16_t* y[kMaxProblems];
  int64_t D[kMaxProblems];
  int cg0[kMaxProblems + 1];         // first channel group of each problem
  int n;
};

template <int VEC, int R, int S, int NC, int MINB, bool SEP>
__global__ void __maxnreg__(regs_for(NC + SEP, MINB))
cconv_fwd_multi_kernel(const __grid_constant__ FwdMulti m) {
  const int cga = blockIdx.x / m.base.cpc;
  int k = 0;
#pragma unroll
  for (int j = 1; j < kMaxProblems; ++j)
    if (j < m.n && cga >= m.cg0[j]) k = j;
  FwdArgs q = m.base;
  q.w = m.w[k];
  q.bias = m.bias[k];
  q.y = m.y[k];
  q.D = m.D[k];
  fwd_cta<VEC, R, S, NC, SEP, 0>(&m.map[k], q, cga - m.cg0[k], blockIdx.x - cga * m.base.cpc);
}

// ------------------------------------------------------------------------------------
// packed sequences: final states (second kernel)
//
// final[slot(i), d, j] = extended row se - (W-1) + j of sequence i: x where that row lies in
// the sequence, else its initial state (zero without one).  One thread per 8 channels of a
// sequence; the 8 channels' W-1 entries are 16*(W-1) contiguous bytes.  It runs after the
// stream kernel has completed (programmatic dependent launch waits for it), so the final
// states may overwrite the initial states in place: every read of them is done by then.
// With state indices it first validates them in every CTA, as the decode update does
// (negative, >= S, or repeated), and on a bad vector writes nothing but the status words.
// ------------------------------------------------------------------------------------
constexpr int kStateThreads = 256;

struct StateArgs {
  const uint16_t* x;      // [total, D], row stride sxt
  const int32_t* cu;      // [nseq + 1]
  const uint16_t* init;   // [S, D, W-1] or null
  uint16_t* fin;          // [S, D, W-1] or null
  const int32_t* idx;     // [nseq] or null
  int32_t* status;        // [2] or null (required with idx)
  int64_t sxt, D, S;
  int nseq, total, chunks;
};

template <int L>
__global__ void __launch_bounds__(kStateThreads) cconv_fwd_state_kernel(const StateArgs p) {
  extern __shared__ uint32_t bitmap[];
  __shared__ int s_bad;
  if (p.idx) {
    if (threadIdx.x == 0) s_bad = 0;
    const int nwords = static_cast<int>((p.S + 31) / 32);
    for (int k = threadIdx.x; k < nwords; k += kStateThreads) bitmap[k] = 0u;
  }
  grid_dependency_wait();
  int bad = 0;
  if (p.idx) {
    __syncthreads();
    int off = 0;
    for (int k = threadIdx.x; k < p.nseq; k += kStateThreads) {
      const int32_t v = p.idx[k];
      if (v < 0) {
        off |= CCONV_IDX_NEGATIVE;
      } else if (v >= p.S) {
        off |= CCONV_IDX_OUT_OF_RANGE;
      } else {
        const uint32_t m = 1u << (v & 31);
        if (atomicOr(&bitmap[v >> 5], m) & m) off |= CCONV_IDX_DUPLICATE;
      }
    }
    if (off) atomicOr(&s_bad, off);
    __syncthreads();
    bad = s_bad;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      p.status[0] = bad ? CCONV_ERR_INDEX : CCONV_OK;
      p.status[1] = bad;
    }
  }
  grid_launch_dependents();
  if (bad || !p.fin || L == 0) return;

  const int64_t items = static_cast<int64_t>(p.nseq) * p.chunks;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kStateThreads + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * kStateThreads) {
    const int i = static_cast<int>(it / p.chunks);
    const int64_t d0 = (it - static_cast<int64_t>(i) * p.chunks) * 8;
    const int64_t slot = p.idx ? p.idx[i] : i;
    const int ss = clamp_row(p.cu[i], p.total);
    int se = clamp_row(p.cu[i + 1], p.total);
    if (se < ss) se = ss;
    uint4 st[L > 0 ? L : 1];  // initial entries of these 8 channels (only if needed)
    const bool short_seq = se - ss < L;
    if (short_seq) {
      if (p.init) {
        const uint4* src = reinterpret_cast<const uint4*>(p.init + (slot * p.D + d0) * L);
#pragma unroll
        for (int u = 0; u < L; ++u) st[u] = src[u];
      } else {
#pragma unroll
        for (int u = 0; u < L; ++u) st[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const uint16_t* sh = reinterpret_cast<const uint16_t*>(st);
    uint4 out[L > 0 ? L : 1];
    uint16_t* oh = reinterpret_cast<uint16_t*>(out);
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const int u = se - L + j;  // extended row
      if (u >= ss) {
        const uint4 v = *reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(u) * p.sxt + d0);
        const uint16_t* vh = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
        for (int c = 0; c < 8; ++c) oh[c * L + j] = vh[c];
      } else {
        const int jj = u - (ss - L);  // entry of the initial state, 0 <= jj < L
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint16_t v = 0;
#pragma unroll
          for (int m = 0; m < L; ++m)  // select in registers (no local-memory indexing)
            if (m == jj) v = sh[c * L + m];
          oh[c * L + j] = v;
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(p.fin + (slot * p.D + d0) * L);
#pragma unroll
    for (int u = 0; u < L; ++u) dst[u] = out[u];
  }
}

// ------------------------------------------------------------------------------------
// launch configuration (a compile-time tile shape)
//
// The product build has one forward tile shape, measured fastest at B=2 T=8192 D=4096.
// Building with -DCCONV_TILE_SWEEP adds the other shapes that were measured against it,
// selected by the environment variable CCONV_FWD_CONFIG (an index into the table); that
// build is for tile sweeps only, and its extra shapes are not covered by the parity tests.
// ------------------------------------------------------------------------------------
struct FwdConfig {
  int vec, rows, stages, nc, ctas_per_sm, sep;
  void (*kernel)(const CUtensorMap, const FwdArgs);
};

#define CCONV_FWD_CFG(V, R, S, NC, M, SEP) \
  FwdConfig { V, R, S, NC, M, SEP, cconv_fwd_kernel<V, R, S, NC, M, SEP, 0> }

static const FwdConfig kFwdConfigs[] = {
    CCONV_FWD_CFG(4, 8, 10, 8, 1, true),
#ifdef CCONV_TILE_SWEEP
    CCONV_FWD_CFG(4, 12, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 16, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 24, 4, 8, 1, true),
    CCONV_FWD_CFG(4, 12, 4, 8, 2, true),
    CCONV_FWD_CFG(8, 8, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 8, 5, 8, 2, false),
    CCONV_FWD_CFG(4, 4, 20, 8, 1, true),
#endif
};

static int fwd_config_index() {
#ifdef CCONV_TILE_SWEEP
  static const int idx = [] {
    constexpr int n = sizeof(kFwdConfigs) / sizeof(kFwdConfigs[0]);
    const char* e = getenv("CCONV_FWD_CONFIG");
    const int v = e ? atoi(e) : 0;
    return (v >= 0 && v < n) ? v : 0;
  }();
  return idx;
#else
  return 0;
#endif
}

}  // namespace cconv

extern "C" CCONV_API int cconv_fwd(const void* x, int64_t B, int64_t T, int64_t D, int64_t sxb,
                                   int64_t sxt, const void* w, const void* bias, cconv_dtype wdt,
                                   int W, void* y, cconv_stream_t stream) {
  using namespace cconv;
  if (!x || !w || !y) return CCONV_ERR_NULL;
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  if (B < 1 || T < 1 || D < 1 || B * T > (int64_t(1) << 31) - 16 || D > (int64_t(1) << 31) - 8)
    return CCONV_ERR_SHAPE;
  if (D % 8 != 0) return CCONV_ERR_ALIGN;
  int rc = check_rows_tensor(x, B, T, D, sxb, sxt);
  if (rc != CCONV_OK) return rc;
  if (reinterpret_cast<uintptr_t>(y) % 16 != 0) return CCONV_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(w) % (wdt == CCONV_F32 ? 4 : 2) != 0) return CCONV_ERR_ALIGN;
  if (bias && reinterpret_cast<uintptr_t>(bias) % (wdt == CCONV_F32 ? 4 : 2) != 0)
    return CCONV_ERR_ALIGN;

  const FwdConfig& cfg = kFwdConfigs[fwd_config_index()];
  int sms = 0;
  rc = sm_count_current_device(&sms, nullptr);
  if (rc != CCONV_OK) return rc;
  const GroupPlan plan = make_group_plan(B, T, D, cfg.vec, cfg.nc, cfg.ctas_per_sm, sms, 32);

  normalise_strides(B, T, D, sxb, sxt);
  CUtensorMap tmx;
  rc = encode_rows_map(&tmx, x, B, T, D, sxb, sxt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;

  FwdArgs a;
  a.w = w;
  a.bias = bias;
  a.y = static_cast<uint16_t*>(y);
  a.D = D;
  a.T = static_cast<int>(T);
  a.BT = static_cast<int>(B * T);
  a.cpc = plan.cpc;
  a.W = W;
  a.wdt = wdt;

  const int stage = cfg.nc * cfg.rows * 32 * cfg.vec * 2;
  const int smem = cfg.stages * (stage + 16);
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(cfg.kernel), smem);
  if (rc != CCONV_OK) return rc;
  return launch_pdl(cfg.kernel, dim3(plan.grid), dim3((cfg.nc + cfg.sep) * 32), smem,
                    reinterpret_cast<cudaStream_t>(stream), tmx, a) == cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}

namespace cconv {

// Packed sequences run the default tile shape (first configuration).
static void (*const kFwdVarlenKernels[2])(const CUtensorMap, const FwdArgs) = {
    cconv_fwd_kernel<4, 8, 10, 8, 1, true, kModeVarlen>,
    cconv_fwd_kernel<4, 8, 10, 8, 1, true, kModeVarlen | kModeActNone>,
};
constexpr int kVarlenVec = 4, kVarlenRows = 8, kVarlenStages = 10, kVarlenNc = 8;

static void (*const kStateKernels[4])(const StateArgs) = {
    cconv_fwd_state_kernel<0>, cconv_fwd_state_kernel<1>, cconv_fwd_state_kernel<2>,
    cconv_fwd_state_kernel<3>};

int launch_index_check(const int32_t* idx, int64_t n, int64_t S, int32_t* status,
                       cudaStream_t stream) {
  StateArgs sa{};
  sa.idx = idx;
  sa.status = status;
  sa.S = S;
  sa.nseq = static_cast<int>(n);
  sa.fin = nullptr;  // validation and status only: one CTA checks every index
  auto kern = kStateKernels[0];
  const size_t smem = static_cast<size_t>((S + 31) / 32) * 4;
  if (smem > 32 * 1024 &&
      set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)) != CCONV_OK)
    return CCONV_ERR_CUDA;
  return launch_pdl(kern, dim3(1), dim3(kStateThreads), smem, stream, sa) == cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}

}  // namespace cconv

extern "C" CCONV_API int cconv_fwd_varlen(const void* x, int64_t total, int64_t D, int64_t sxt,
                                          const int32_t* cu_seqlens, int64_t nseq,
                                          const void* w, const void* bias, cconv_dtype wdt,
                                          int W, cconv_activation act,
                                          const void* initial_state, void* final_state,
                                          const int32_t* state_indices, int64_t S,
                                          int32_t* status_dev, void* y, cconv_stream_t stream) {
  using namespace cconv;
  if (!w || !cu_seqlens) return CCONV_ERR_NULL;
  if (total > 0 && (!x || !y)) return CCONV_ERR_NULL;
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  if (act != CCONV_ACT_SILU && act != CCONV_ACT_NONE) return CCONV_ERR_SHAPE;
  if (total < 0 || nseq < 1 || D < 1 || total > (int64_t(1) << 31) - 16 ||
      nseq > (int64_t(1) << 31) - 2 || D > (int64_t(1) << 31) - 8)
    return CCONV_ERR_SHAPE;
  if (D % 8 != 0) return CCONV_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(cu_seqlens) % 4 != 0) return CCONV_ERR_ALIGN;
  int rc;
  if (total > 0) {
    rc = check_rows_tensor(x, 1, total, D, 0, sxt);
    if (rc != CCONV_OK) return rc;
    if (reinterpret_cast<uintptr_t>(y) % 16 != 0) return CCONV_ERR_ALIGN;
  }
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(w) % ew != 0 ||
      (bias && reinterpret_cast<uintptr_t>(bias) % ew != 0))
    return CCONV_ERR_ALIGN;
  const int L = W - 1;
  const bool states = L > 0 && (initial_state || final_state);
  if (state_indices) {
    if (!status_dev) return CCONV_ERR_NULL;
    if (S < 1 || S > CCONV_UPDATE_MAX_SLOTS) return CCONV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(state_indices) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(status_dev) % 4 != 0)
      return CCONV_ERR_ALIGN;
  } else if (states && S < nseq) {
    return CCONV_ERR_SHAPE;
  }
  if (states && ((initial_state && reinterpret_cast<uintptr_t>(initial_state) % 16 != 0) ||
                 (final_state && reinterpret_cast<uintptr_t>(final_state) % 16 != 0)))
    return CCONV_ERR_ALIGN;

  // Dense final states that do not overlap the initial states are written by the stream
  // kernel itself, from its register ring; slots picked by state_indices (validated first)
  // or states updated in place need the second kernel, which runs after every read.
  const size_t state_bytes = static_cast<size_t>(nseq) * D * (L > 0 ? L : 1) * 2;
  const uintptr_t ib = reinterpret_cast<uintptr_t>(initial_state);
  const uintptr_t fb = reinterpret_cast<uintptr_t>(final_state);
  const bool overlap = initial_state && final_state && ib < fb + state_bytes && fb < ib + state_bytes;
  const bool fused_final = L > 0 && final_state && !state_indices && !overlap && total > 0;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (total > 0) {
    int sms = 0;
    rc = sm_count_current_device(&sms, nullptr);
    if (rc != CCONV_OK) return rc;
    const GroupPlan plan =
        make_group_plan(1, total, D, kVarlenVec, kVarlenNc, 1, sms, 32);
    int64_t sb = 0;
    normalise_strides(1, total, D, sb, sxt);
    CUtensorMap tmx;
    rc = encode_rows_map(&tmx, x, 1, total, D, sb, sxt, 32 * kVarlenVec, kVarlenRows);
    if (rc != CCONV_OK) return rc;
    FwdArgs a;
    a.w = w;
    a.bias = bias;
    a.y = static_cast<uint16_t*>(y);
    a.D = D;
    a.T = static_cast<int>(total);
    a.BT = static_cast<int>(total);
    a.cpc = plan.cpc;
    a.W = W;
    a.wdt = wdt;
    a.cu = cu_seqlens;
    a.init = L > 0 ? static_cast<const uint16_t*>(initial_state) : nullptr;
    a.idx = state_indices;
    a.fin = fused_final ? static_cast<uint16_t*>(final_state) : nullptr;
    a.S = state_indices ? S : nseq;
    a.nseq = static_cast<int>(nseq);
    auto kern = kFwdVarlenKernels[act == CCONV_ACT_NONE ? 1 : 0];
    const int smem = kVarlenStages * (kVarlenNc * kVarlenRows * 32 * kVarlenVec * 2 + 16);
    rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (rc != CCONV_OK) return rc;
    if (launch_pdl(kern, dim3(plan.grid), dim3((kVarlenNc + 1) * 32), smem, st, tmx, a) !=
        cudaSuccess)
      return CCONV_ERR_CUDA;
  }
  if ((L > 0 && final_state && !fused_final) || state_indices) {
    int sms = 0;
    rc = sm_count_current_device(&sms, nullptr);
    if (rc != CCONV_OK) return rc;
    StateArgs sa;
    sa.x = static_cast<const uint16_t*>(x);
    sa.cu = cu_seqlens;
    sa.init = L > 0 ? static_cast<const uint16_t*>(initial_state) : nullptr;
    sa.fin = L > 0 ? static_cast<uint16_t*>(final_state) : nullptr;
    sa.idx = state_indices;
    sa.status = status_dev;
    sa.sxt = sxt;
    sa.D = D;
    sa.S = state_indices ? S : nseq;
    sa.nseq = static_cast<int>(nseq);
    sa.total = static_cast<int>(total);
    sa.chunks = static_cast<int>(D / 8);
    const int64_t items = nseq * (D / 8);
    int64_t grid = (items + kStateThreads - 1) / kStateThreads;
    if (grid > 2 * sms) grid = 2 * sms;
    if (grid < 1) grid = 1;
    auto kern = kStateKernels[L];
    const size_t smem = state_indices ? static_cast<size_t>((S + 31) / 32) * 4 : 0;
    if (smem > 32 * 1024 &&
        set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)) != CCONV_OK)
      return CCONV_ERR_CUDA;
    if (launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kStateThreads), smem, st, sa) !=
        cudaSuccess)
      return CCONV_ERR_CUDA;
  }
  return CCONV_OK;
}

extern "C" CCONV_API int cconv_fwd_multi(int n, const void* const* x, const int64_t* D,
                                         const int64_t* sxb, const int64_t* sxt,
                                         const void* const* w, const void* const* bias,
                                         void* const* y, int64_t B, int64_t T, cconv_dtype wdt,
                                         int W, cconv_stream_t stream) {
  using namespace cconv;
  if (!x || !D || !sxb || !sxt || !w || !y) return CCONV_ERR_NULL;
  if (n < 1 || n > kMaxProblems) return CCONV_ERR_SHAPE;
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  if (B < 1 || T < 1 || B * T > (int64_t(1) << 31) - 16) return CCONV_ERR_SHAPE;
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  constexpr int kVec = 4, kRows = 8, kStages = 10, kNc = 8;
  constexpr int64_t kGroup = int64_t(kNc) * 32 * kVec;
  FwdMulti m;
  int cg_total = 0;
  for (int k = 0; k < n; ++k) {
    const void* bk = bias ? bias[k] : nullptr;
    if (!x[k] || !w[k] || !y[k]) return CCONV_ERR_NULL;
    if (D[k] < 1 || D[k] > (int64_t(1) << 31) - 8) return CCONV_ERR_SHAPE;
    if (D[k] % 8 != 0) return CCONV_ERR_ALIGN;
    int rc = check_rows_tensor(x[k], B, T, D[k], sxb[k], sxt[k]);
    if (rc != CCONV_OK) return rc;
    if (reinterpret_cast<uintptr_t>(y[k]) % 16 != 0) return CCONV_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(w[k]) % ew != 0 ||
        (bk && reinterpret_cast<uintptr_t>(bk) % ew != 0))
      return CCONV_ERR_ALIGN;
    m.cg0[k] = cg_total;
    cg_total += static_cast<int>((D[k] + kGroup - 1) / kGroup);
  }
  m.cg0[n] = cg_total;
  int sms = 0;
  int rc = sm_count_current_device(&sms, nullptr);
  if (rc != CCONV_OK) return rc;
  int64_t cpc = sms / cg_total;
  if (cpc < 1) cpc = 1;
  const int64_t by_rows = (B * T) / 32 > 0 ? (B * T) / 32 : 1;
  if (cpc > by_rows) cpc = by_rows;
  for (int k = 0; k < n; ++k) {
    int64_t sb = sxb[k], st = sxt[k];
    normalise_strides(B, T, D[k], sb, st);
    rc = encode_rows_map(&m.map[k], x[k], B, T, D[k], sb, st, 32 * kVec, kRows);
    if (rc != CCONV_OK) return rc;
    m.w[k] = w[k];
    m.bias[k] = bias ? bias[k] : nullptr;
    m.y[k] = static_cast<uint16_t*>(y[k]);
    m.D[k] = D[k];
  }
  for (int k = n; k < kMaxProblems; ++k) {  // unused slots: copies of the last problem
    m.map[k] = m.map[n - 1];
    m.w[k] = m.w[n - 1];
    m.bias[k] = m.bias[n - 1];
    m.y[k] = m.y[n - 1];
    m.D[k] = m.D[n - 1];
    m.cg0[k + 1 > kMaxProblems ? kMaxProblems : k + 1] = cg_total;
  }
  m.n = n;
  FwdArgs& a = m.base;
  a = FwdArgs{};
  a.T = static_cast<int>(T);
  a.BT = static_cast<int>(B * T);
  a.cpc = static_cast<int>(cpc);
  a.W = W;
  a.wdt = wdt;
  auto kern = cconv_fwd_multi_kernel<kVec, kRows, kStages, kNc, 1, true>;
  const int smem = kStages * (kNc * kRows * 32 * kVec * 2 + 16);
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
  if (rc != CCONV_OK) return rc;
  return launch_pdl(kern, dim3(static_cast<unsigned>(cg_total * cpc)), dim3((kNc + 1) * 32), smem,
                    reinterpret_cast<cudaStream_t>(stream), m) == cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}
