// update.cu -- cconv_update / cconv_update_ex: single-token decode update of a pooled conv
// state (one kernel).
//
// Per row i with slot s = state_indices[i] (or i):
//   window     = (state[s,d,0..W-2], x[i,d])          state[...,0] is the oldest
//   y[i,d]     = silu(bias[d] + sum_{j<W} w[d,j] * window[j])
//   state[s,d] = window[1..W-1]                        (bf16 bits copied exactly)
// Source: "Add experimental causal conv1d decode update - #797" (NVIDIA/cudnn-frontend),
// PR summary; the forward's tap orientation (kernel-fun 0.2.0.dev1 wheel,
// cconv/_kernels/strip.py `_tap`) fixes which tap meets which window entry.
//
// Index validation is fused and fails closed without a trap: every CTA loads all N
// indices, range-checks them and finds repeats with a one-bit-per-slot bitmap in shared
// memory, so all CTAs reach the same verdict with no inter-CTA communication.  On a bad
// vector no CTA writes anything but CTA 0's status words (state rows are only read, and
// only for in-range slots).  This replaces the pages' per-CTA O(N^2) scan and device trap
// with an O(N + S/32) check and a status word.
//
// cconv_update_ex runs the same kernel with the PR's variants: a state of L = W entries
// (the window takes the newest W-1), -1 as a padding row, circular-buffer states (the token
// goes to entry cache_seqlens[i] mod L and nothing shifts), and no activation.
#include <algorithm>
#include <cstdlib>

#include "common.cuh"

namespace cconv {

// Shared memory per SM and the amount reserved per block on the current device (cached;
// defined in host.cu).
int smem_per_sm_current_device(int* per_sm, int* reserved_per_block);

struct UpdArgs {
  const uint16_t* x;  // [N, ldx]
  uint16_t* state;    // [S, D, L]
  const int32_t* idx; // [N] or null
  const void* w;      // [D, W]
  const void* bias;   // [D] or null
  uint16_t* y;        // [N, D]
  int32_t* status;    // [2]
  int64_t N, D, ldx, S;
  int wdt;
  int pad;            // nonzero: index -1 marks a padding row
  int act;            // CCONV_ACT_SILU or CCONV_ACT_NONE
  const int32_t* pos; // [N] circular-buffer positions (ring mode), or null
  int64_t gq;         // row lanes: N / gridDim.y rows per group, plus one for the first
  int64_t grem;       //   N % gridDim.y groups
};

// Kernel modes: the plain decode call; the general one (padding rows, activation read from
// the arguments); the general one on circular-buffer states.
enum : int { kUpdPlain = 0, kUpdGeneral = 1, kUpdRing = 2 };

__device__ __forceinline__ int ring_mod(int64_t a, int m) {
  const int r = static_cast<int>(a % m);
  return r < 0 ? r + m : r;
}

// Threads per CTA: 256, or 64 for small decode batches on the vector path (more CTAs over
// the same rows; the host picks).
constexpr int kUpdThreads = 256;
constexpr int kUpdThreadsSmall = 64;

__device__ __forceinline__ float load_w(const void* p, int64_t i, int wdt) {
  return wdt == CCONV_F32 ? static_cast<const float*>(p)[i]
                          : bf16_to_f32(static_cast<const uint16_t*>(p)[i]);
}

__device__ __forceinline__ float silu_f(float z) {
  return z * fmaf(tanh_approx(0.5f * z), 0.5f, 0.5f);
}

// Taps w[d0..d0+VEC-1][0..W-1] and bias of VEC consecutive channels.  The vector path
// (VEC = 8) reads them as 16-byte runs: 8 channels x W taps are 32*W contiguous bytes in
// fp32 (16*W in bf16), and the host only picks it when w and bias are 16-byte aligned.
template <int VEC, int W>
__device__ __forceinline__ void load_update_taps(const UpdArgs& p, int64_t d0,
                                                 float (&tw)[VEC][W], float (&tb)[VEC]) {
  if constexpr (VEC == 8) {
    if (p.wdt == CCONV_F32) {
      float4 v[2 * W];
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.w) + d0 * W);
#pragma unroll
      for (int u = 0; u < 2 * W; ++u) v[u] = src[u];
      const float* f = reinterpret_cast<const float*>(v);
#pragma unroll
      for (int c = 0; c < VEC; ++c)
#pragma unroll
        for (int j = 0; j < W; ++j) tw[c][j] = f[c * W + j];
    } else {
      uint4 v[W];
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.w) + d0 * W);
#pragma unroll
      for (int u = 0; u < W; ++u) v[u] = src[u];
      const uint16_t* h = reinterpret_cast<const uint16_t*>(v);
#pragma unroll
      for (int c = 0; c < VEC; ++c)
#pragma unroll
        for (int j = 0; j < W; ++j) tw[c][j] = bf16_to_f32(h[c * W + j]);
    }
    if (!p.bias) {
#pragma unroll
      for (int c = 0; c < VEC; ++c) tb[c] = 0.f;
    } else if (p.wdt == CCONV_F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.bias) + d0);
      const float4 b0 = src[0], b1 = src[1];
      tb[0] = b0.x; tb[1] = b0.y; tb[2] = b0.z; tb[3] = b0.w;
      tb[4] = b1.x; tb[5] = b1.y; tb[6] = b1.z; tb[7] = b1.w;
    } else {
      const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.bias) + d0);
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&b);
#pragma unroll
      for (int c = 0; c < VEC; ++c) tb[c] = bf16_to_f32(h[c]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
#pragma unroll
      for (int j = 0; j < W; ++j) tw[c][j] = load_w(p.w, (d0 + c) * W + j, p.wdt);
      tb[c] = p.bias ? load_w(p.bias, d0 + c, p.wdt) : 0.f;
    }
  }
}

// Taps and bias of a CTA that covers CV channel vectors (8 channels each) with several row
// lanes: the CTA copies them once into shared memory and every row lane reads them there,
// so only the few CTAs of one channel block, not every row group, fetch the same taps from
// L2.  16-byte unit u of channel vector c sits at tap_s[u * CV + c] (taps first, then the
// bias), so the warp that reads unit u of 32 consecutive channel vectors hits 32 consecutive
// units without bank conflicts.  A channel vector holds 2W tap units and 2 bias units in
// fp32, W and 1 in bf16.
template <int W, int CV>
constexpr int kTapUnits = CV * 2 * (W + 1);

template <int W, int CV, int NT>
struct TapStage {
  static constexpr int K = (kTapUnits<W, CV> + NT - 1) / NT;
  uint4 v[K];
  int dst[K];  // destination unit in shared memory, -1 for nothing
};

// Issue this thread's share of the copy (global loads into registers only).
template <int W, int CV, int NT>
__device__ __forceinline__ void tap_stage_load(const UpdArgs& p, int64_t cv0, int64_t nvec,
                                               TapStage<W, CV, NT>& t) {
  const bool f32 = p.wdt == CCONV_F32;
  const int uw = f32 ? 2 * W : W;  // tap units per channel vector
  const int ub = f32 ? 2 : 1;      // bias units per channel vector
  const int cvs = static_cast<int>(nvec - cv0 < CV ? nvec - cv0 : CV);
  const int ntap = cvs * uw, nall = p.bias ? cvs * (uw + ub) : ntap;
  const int esz = f32 ? 4 : 2;
  const uint4* wsrc = reinterpret_cast<const uint4*>(static_cast<const char*>(p.w) +
                                                     cv0 * 8 * W * esz);
  const uint4* bsrc = p.bias ? reinterpret_cast<const uint4*>(
                                   static_cast<const char*>(p.bias) + cv0 * 8 * esz)
                             : nullptr;
#pragma unroll
  for (int k = 0; k < TapStage<W, CV, NT>::K; ++k) {
    const int g = threadIdx.x + k * NT;
    t.dst[k] = -1;
    if (g < ntap) {
      const int c = f32 ? g / (2 * W) : g / W, u = g - c * uw;
      t.v[k] = wsrc[g];
      t.dst[k] = u * CV + c;
    } else if (g < nall) {
      const int h = g - ntap;
      const int c = f32 ? h >> 1 : h, u = uw + (h - c * ub);
      t.v[k] = bsrc[h];
      t.dst[k] = u * CV + c;
    }
  }
}

template <int W, int CV, int NT>
__device__ __forceinline__ void tap_stage_store(uint4* tap_s, const TapStage<W, CV, NT>& t) {
#pragma unroll
  for (int k = 0; k < TapStage<W, CV, NT>::K; ++k)
    if (t.dst[k] >= 0) tap_s[t.dst[k]] = t.v[k];
}

// Channel vector c's taps and bias from the staged copy (visible after a barrier).
template <int W, int CV>
__device__ __forceinline__ void tap_stage_read(const UpdArgs& p, const uint4* tap_s, int c,
                                               float (&tw)[8][W], float (&tb)[8]) {
  if (p.wdt == CCONV_F32) {
    float4 v[2 * W];
#pragma unroll
    for (int u = 0; u < 2 * W; ++u) v[u] = *reinterpret_cast<const float4*>(&tap_s[u * CV + c]);
    const float* f = reinterpret_cast<const float*>(v);
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int j = 0; j < W; ++j) tw[k][j] = f[k * W + j];
    if (p.bias) {
      const float4 b0 = *reinterpret_cast<const float4*>(&tap_s[2 * W * CV + c]);
      const float4 b1 = *reinterpret_cast<const float4*>(&tap_s[(2 * W + 1) * CV + c]);
      tb[0] = b0.x; tb[1] = b0.y; tb[2] = b0.z; tb[3] = b0.w;
      tb[4] = b1.x; tb[5] = b1.y; tb[6] = b1.z; tb[7] = b1.w;
    }
  } else {
    uint4 v[W];
#pragma unroll
    for (int u = 0; u < W; ++u) v[u] = tap_s[u * CV + c];
    const uint16_t* h = reinterpret_cast<const uint16_t*>(v);
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int j = 0; j < W; ++j) tw[k][j] = bf16_to_f32(h[k * W + j]);
    if (p.bias) {
      const uint4 b = tap_s[W * CV + c];
      const uint16_t* bh = reinterpret_cast<const uint16_t*>(&b);
#pragma unroll
      for (int k = 0; k < 8; ++k) tb[k] = bf16_to_f32(bh[k]);
    }
  }
  if (!p.bias) {
#pragma unroll
    for (int k = 0; k < 8; ++k) tb[k] = 0.f;
  }
}

// Channel vectors per CTA row lane: the 256-thread vector kernels run 32 channel vectors x 8
// row lanes; the others give every thread of a CTA its own channel vector (one row lane).
template <int VEC, int NT>
__host__ __device__ constexpr int update_cv() { return (VEC == 8 && NT == 256) ? 32 : NT; }

// VEC = channels per thread (8: 16-byte vectors; 1: scalar path), W taps, L = state entries
// per channel (W - 1, or W to keep one older token: the newest W - 1 feed the window, and
// the new state is the last L of (old state, token), i.e. window[W - L + j]), ROWS = rows
// per thread.  A CTA is CV channel vectors x RL = NT / CV row lanes; grid x over blocks of CV
// channel vectors, y over row groups.  With one row lane a group is ROWS consecutive rows.
// With several, the N rows are split evenly over gridDim.y groups of at most RL * ROWS rows
// (the first N % gridDim.y groups one row longer)
// (so the host can size the grid to the SM count), lane l takes rows l, l + RL, ... of its
// group, and the CTA stages its taps in shared memory once.
//
// Latency is what this kernel is about (a decode step moves ~17 MB, mostly L2-resident), so
// every independent load is issued before the index check needs to finish: this thread's
// slot ids, token rows, taps and bias first, then the CTA's pass over all N indices; the
// state rows of in-range slots are fetched while the check completes.  Only the writes wait
// for the verdict.  Padding rows (p.pad, index -1) are left out of the check and touch
// neither the state nor y.  MODE kUpdGeneral: the padding mode and the activation are read
// from p; kUpdPlain fixes them to "off" and SiLU at compile time (the plain decode call,
// whose latency the runtime tests measurably add to).  kUpdRing: the state of a slot is a
// ring of L entries; the token goes to entry head = pos[i] mod L, the window is the W-1
// entries before it (oldest first), and only the head entry is written.
template <int VEC, int W, int L, int ROWS, int MODE, int NT>
__global__ void __launch_bounds__(NT) cconv_update_kernel(const UpdArgs p) {
  static_assert(L == W - 1 || L == W, "state length is W-1 or W");
  static_assert(MODE != kUpdRing || L > 0, "a ring needs at least one entry");
  constexpr bool GEN = MODE != kUpdPlain;
  constexpr bool RING = MODE == kUpdRing;
  constexpr int OFF = L - (W - 1);  // state entries older than the window (0 or 1)
  const bool pad = GEN && p.pad != 0;
  const bool act_none = GEN && p.act == CCONV_ACT_NONE;
  constexpr int CV = update_cv<VEC, NT>();
  constexpr int RL = NT / CV;
  static_assert(RL * CV == NT && (RL == 1 || VEC == 8), "row lanes need the vector path");
  extern __shared__ uint32_t bitmap[];
  __shared__ int s_bad;
  __shared__ uint4 tap_s[RL > 1 ? kTapUnits<W, CV> : 1];

  if (p.idx) {  // shared-memory set-up only: no global access before the dependency wait
    if (threadIdx.x == 0) s_bad = 0;
    const int nwords = static_cast<int>((p.S + 31) / 32);
    for (int i = threadIdx.x; i < nwords; i += NT) bitmap[i] = 0u;
  }
  grid_dependency_wait();

  const int cl = RL > 1 ? static_cast<int>(threadIdx.x % CV) : static_cast<int>(threadIdx.x);
  const int rl = RL > 1 ? static_cast<int>(threadIdx.x / CV) : 0;
  const int64_t cv0 = static_cast<int64_t>(blockIdx.x) * CV;
  const int64_t d0 = (cv0 + cl) * VEC;
  const bool mine = d0 < p.D;
  // rows of this thread: row_of(r) for r < ROWS, valid while below iend
  const int64_t by = blockIdx.y;
  const int64_t ib = RL > 1 ? p.gq * by + (by < p.grem ? by : p.grem) : by * ROWS;
  const int64_t iend = RL > 1 ? ib + p.gq + (by < p.grem ? 1 : 0) : p.N;
  auto row_of = [&](int r) -> int64_t { return ib + static_cast<int64_t>(r) * RL + rl; };

  // ---- this thread's rows: slot ids, token rows, taps ------------------------------------
  // slot[r] < 0: no row, or a padding row (nothing to do for it)
  int64_t slot[ROWS];
  int head[ROWS];  // ring mode: the entry the token goes to
  uint16_t win[ROWS][VEC][W];
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    const int64_t i = row_of(r);
    slot[r] = (mine && i < iend) ? (p.idx ? static_cast<int64_t>(p.idx[i]) : i) : -1;
    if constexpr (RING) head[r] = (mine && i < iend) ? ring_mod(p.pos[i], L) : 0;
    if (pad && slot[r] == -1) continue;
    if (mine && i < iend) {
      const uint16_t* xr = p.x + i * p.ldx + d0;
      if constexpr (VEC == 8) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xr);
        const uint16_t* xh = reinterpret_cast<const uint16_t*>(&xv);
#pragma unroll
        for (int c = 0; c < VEC; ++c) win[r][c][W - 1] = xh[c];
      } else {
        win[r][0][W - 1] = xr[0];
      }
    }
  }
  float tw[VEC][W], tb[VEC];
  TapStage<W, CV, NT> stage;
  if constexpr (RL > 1)
    tap_stage_load<W, CV, NT>(p, cv0, (p.D + VEC - 1) / VEC, stage);
  else if (mine)
    load_update_taps<VEC, W>(p, d0, tw, tb);

  // ---- validation: identical verdict in every CTA --------------------------------------
  int bad = 0;
  if (p.idx) {
    __syncthreads();  // the zeroed bitmap is visible
    int off = 0;
    for (int64_t i = threadIdx.x; i < p.N; i += NT) {
      const int32_t v = p.idx[i];
      if (pad && v == -1) continue;  // a padding row
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
  }

  // ---- state rows of in-range slots, fetched while the check completes ------------------
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    if (slot[r] < 0 || slot[r] >= p.S) continue;
    const uint16_t* st = p.state + (slot[r] * p.D + d0) * L;
    if constexpr (VEC == 8) {
      // 8 channels x L state entries are 16*L contiguous bytes
      uint4 sv[L > 0 ? L : 1];
#pragma unroll
      for (int u = 0; u < L; ++u) sv[u] = reinterpret_cast<const uint4*>(st)[u];
      const uint16_t* sh = reinterpret_cast<const uint16_t*>(sv);
      if constexpr (RING) {
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
          const int e = ring_mod(head[r] - (W - 1) + j, L);
#pragma unroll
          for (int c = 0; c < VEC; ++c) {
            uint16_t v = 0;
#pragma unroll
            for (int m = 0; m < L; ++m)  // select in registers (no local-memory indexing)
              if (m == e) v = sh[c * L + m];
            win[r][c][j] = v;
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < VEC; ++c)
#pragma unroll
          for (int j = 0; j < W - 1; ++j) win[r][c][j] = sh[c * L + OFF + j];
      }
    } else if constexpr (RING) {
#pragma unroll
      for (int j = 0; j < W - 1; ++j) win[r][0][j] = st[ring_mod(head[r] - (W - 1) + j, L)];
    } else {
#pragma unroll
      for (int j = 0; j < W - 1; ++j) win[r][0][j] = st[OFF + j];
    }
  }

  if constexpr (RL > 1) tap_stage_store<W, CV, NT>(tap_s, stage);
  if (p.idx || RL > 1) {
    __syncthreads();  // every index of this CTA's pass is checked; the staged taps are visible
    if (p.idx) bad = s_bad;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    p.status[0] = bad ? CCONV_ERR_INDEX : CCONV_OK;
    p.status[1] = bad;
  }
  grid_launch_dependents();
  if (bad || !mine) return;
  if constexpr (RL > 1) tap_stage_read<W, CV>(p, tap_s, cl, tw, tb);

  // ---- y and the shifted state (writes only after a clean verdict) -----------------------
#pragma unroll
  for (int r = 0; r < ROWS; ++r) {
    if (slot[r] < 0) continue;
    uint16_t yo[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
      float z = tb[c];
#pragma unroll
      for (int j = 0; j < W; ++j) z = fmaf(tw[c][j], bf16_to_f32(win[r][c][j]), z);
      yo[c] = f32_to_bf16(act_none ? z : silu_f(z));
    }
    uint16_t* st = p.state + (slot[r] * p.D + d0) * L;
    uint16_t* yr = p.y + row_of(r) * p.D + d0;
    if constexpr (RING) {
      if constexpr (VEC == 8)
        *reinterpret_cast<uint4*>(yr) = *reinterpret_cast<const uint4*>(yo);
      else
        yr[0] = yo[0];
#pragma unroll
      for (int c = 0; c < VEC; ++c) st[c * L + head[r]] = win[r][c][W - 1];  // the token
    } else if constexpr (VEC == 8) {
      *reinterpret_cast<uint4*>(yr) = *reinterpret_cast<const uint4*>(yo);
      if constexpr (L > 0) {
        uint4 nv[L];
        uint16_t* nh = reinterpret_cast<uint16_t*>(nv);
#pragma unroll
        for (int c = 0; c < VEC; ++c)
#pragma unroll
          for (int j = 0; j < L; ++j) nh[c * L + j] = win[r][c][W - L + j];
#pragma unroll
        for (int u = 0; u < L; ++u) reinterpret_cast<uint4*>(st)[u] = nv[u];
      }
    } else {
      yr[0] = yo[0];
#pragma unroll
      for (int j = 0; j < L; ++j) st[j] = win[r][0][W - L + j];
    }
  }
}

typedef void (*UpdKernel)(const UpdArgs);

// No kernel for a ring of zero entries (the host refuses it before choosing).
template <int VEC, int W, int L, int ROWS, int MODE, int NT>
static UpdKernel update_kernel() {
  if constexpr (MODE == kUpdRing && L == 0)
    return nullptr;
  else
    return cconv_update_kernel<VEC, W, L, ROWS, MODE, NT>;
}

template <int VEC, int ROWS, int OFF, int MODE, int NT>
static UpdKernel pick_update_kernel_w(int W) {
  switch (W) {
    case 1: return update_kernel<VEC, 1, 0 + OFF, ROWS, MODE, NT>();
    case 2: return update_kernel<VEC, 2, 1 + OFF, ROWS, MODE, NT>();
    case 3: return update_kernel<VEC, 3, 2 + OFF, ROWS, MODE, NT>();
    default: return update_kernel<VEC, 4, 3 + OFF, ROWS, MODE, NT>();
  }
}

// L = W - 1 + off.  mode: kUpdGeneral when padding rows or another activation are asked
// for, kUpdRing for circular-buffer states.  The general kernels take fewer row counts (1
// and 4), and the 64-thread plain kernels 1, 2 and 4.
template <int VEC, int NT>
static UpdKernel pick_update_kernel(int W, int rows, int off, int mode) {
  if (mode == kUpdRing) {
    if (off)
      return rows >= 4 ? pick_update_kernel_w<VEC, 4, 1, kUpdRing, NT>(W)
                       : pick_update_kernel_w<VEC, 1, 1, kUpdRing, NT>(W);
    return rows >= 4 ? pick_update_kernel_w<VEC, 4, 0, kUpdRing, NT>(W)
                     : pick_update_kernel_w<VEC, 1, 0, kUpdRing, NT>(W);
  }
  if (off || mode == kUpdGeneral) {
    if (off)
      return rows >= 4 ? pick_update_kernel_w<VEC, 4, 1, kUpdGeneral, NT>(W)
                       : pick_update_kernel_w<VEC, 1, 1, kUpdGeneral, NT>(W);
    return rows >= 4 ? pick_update_kernel_w<VEC, 4, 0, kUpdGeneral, NT>(W)
                     : pick_update_kernel_w<VEC, 1, 0, kUpdGeneral, NT>(W);
  }
  if constexpr (NT == kUpdThreadsSmall) {
    switch (rows) {
      case 1: return pick_update_kernel_w<VEC, 1, 0, kUpdPlain, NT>(W);
      case 2: return pick_update_kernel_w<VEC, 2, 0, kUpdPlain, NT>(W);
      default: return pick_update_kernel_w<VEC, 4, 0, kUpdPlain, NT>(W);
    }
  } else {
    switch (rows) {
      case 1: return pick_update_kernel_w<VEC, 1, 0, kUpdPlain, NT>(W);
      case 2: return pick_update_kernel_w<VEC, 2, 0, kUpdPlain, NT>(W);
#ifdef CCONV_TILE_SWEEP
      case 8: return pick_update_kernel_w<VEC, 8, 0, kUpdPlain, NT>(W);
      case 16: return pick_update_kernel_w<VEC, 16, 0, kUpdPlain, NT>(W);
#endif
      default: return pick_update_kernel_w<VEC, 4, 0, kUpdPlain, NT>(W);
    }
  }
}

// The decode update with every option: state length L (W - 1 or W), padding rows, activation.
static int update_impl(const void* x, int64_t N, int64_t D, int64_t ldx, void* state, int64_t S,
                       int L, const int32_t* state_indices, int pad, const int32_t* pos,
                       const void* w, const void* bias, cconv_dtype wdt, int W,
                       cconv_activation act, void* y, int32_t* status_dev,
                       cconv_stream_t stream) {
  if (!x || !w || !y || !status_dev) return CCONV_ERR_NULL;
  if (W < 1 || W > 4) return CCONV_ERR_WIDTH;
  if (L != W - 1 && L != W) return CCONV_ERR_SHAPE;
  if (pos && L < 1) return CCONV_ERR_SHAPE;  // a ring needs at least one entry
  if (pos && reinterpret_cast<uintptr_t>(pos) % 4 != 0) return CCONV_ERR_ALIGN;
  if (act != CCONV_ACT_SILU && act != CCONV_ACT_NONE) return CCONV_ERR_SHAPE;
  if (L > 0 && !state) return CCONV_ERR_NULL;
  if (wdt != CCONV_BF16 && wdt != CCONV_F32) return CCONV_ERR_DTYPE;
  if (N < 1 || D < 1 || S < 0 || N > (int64_t(1) << 31) - 1 || D > (int64_t(1) << 31) - 8)
    return CCONV_ERR_SHAPE;
  if (ldx < D) return CCONV_ERR_STRIDE;
  if (state_indices) {
    if (S > CCONV_UPDATE_MAX_SLOTS) return CCONV_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(state_indices) % 4 != 0) return CCONV_ERR_ALIGN;
  } else if (S < N) {
    return CCONV_ERR_SHAPE;
  }
  const int ew = wdt == CCONV_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(w) % ew != 0 ||
      (bias && reinterpret_cast<uintptr_t>(bias) % ew != 0))
    return CCONV_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(x) % 2 != 0 || reinterpret_cast<uintptr_t>(y) % 2 != 0 ||
      (state && reinterpret_cast<uintptr_t>(state) % 2 != 0) ||
      reinterpret_cast<uintptr_t>(status_dev) % 4 != 0)
    return CCONV_ERR_ALIGN;

  const int ew16 = 16;
  const bool vec8 = D % 8 == 0 && ldx % 8 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
                    (!state || reinterpret_cast<uintptr_t>(state) % 16 == 0) &&
                    reinterpret_cast<uintptr_t>(w) % ew16 == 0 &&
                    (!bias || reinterpret_cast<uintptr_t>(bias) % ew16 == 0);
  const int vec = vec8 ? 8 : 1;

  int sms = 0;
  int rc = sm_count_current_device(&sms, nullptr);
  if (rc != CCONV_OK) return rc;
  const int off = L - (W - 1);
  const int mode = pos ? kUpdRing : (pad != 0 || act != CCONV_ACT_SILU) ? kUpdGeneral : kUpdPlain;
  const int64_t nvec = (D + vec - 1) / vec;
  // Small batches on the vector path: 64-thread CTAs (one row lane), when one or two rows
  // per thread keep their grid within one wave; otherwise the 256-thread CTAs (8 row lanes
  // sharing staged taps).  Measured in CUDA graphs at S=512 W=4, us per step, 64- against
  // 256-thread CTAs: D=1024 N=64 1.95 / 2.17 and N=192 2.94 / 2.16; D=2048 N=64 2.03 / 2.22
  // and N=128 2.67 / 2.22; D=4096 N=16 1.78 / 2.25 and N=64 2.46 / 2.18; D=8192 N=16
  // 1.96 / 2.29 and N=64 3.24 / 2.79.
  int nt = kUpdThreads;
  int rows = 4;
  if (vec == 8) {
    const int64_t gx_small = (nvec + kUpdThreadsSmall - 1) / kUpdThreadsSmall;
    for (int r = 1; r <= 2; r *= 2) {
      if (gx_small * ((N + r - 1) / r) <= sms) {
        nt = kUpdThreadsSmall;
        rows = r;
        break;
      }
    }
  }
#ifdef CCONV_TILE_SWEEP
  // CCONV_UPDATE_THREADS=256 or 64 picks the CTA size on the vector path.
  static const int threads_override = [] {
    const char* e = getenv("CCONV_UPDATE_THREADS");
    const int v = e ? atoi(e) : 0;
    return (v == kUpdThreads || v == kUpdThreadsSmall) ? v : 0;
  }();
  if (vec == 8 && threads_override == kUpdThreads && nt != kUpdThreads) {
    nt = kUpdThreads;
    rows = 4;
  } else if (vec == 8 && threads_override == kUpdThreadsSmall && nt != kUpdThreadsSmall) {
    const int64_t gx_small = (nvec + kUpdThreadsSmall - 1) / kUpdThreadsSmall;
    int r = 1;
    while (r < 4 && gx_small * ((N + r - 1) / r) > sms) r *= 2;
    nt = kUpdThreadsSmall;
    rows = r;
  }
#endif
  // Channel vectors per CTA and row lanes (the kernels' own split, update_cv).
  const int cv = (vec == 8 && nt == kUpdThreads) ? update_cv<8, kUpdThreads>() : nt;
  const int rl = nt / cv;
  const int64_t gx = (nvec + cv - 1) / cv;
  if (nt == kUpdThreads) {
    // Rows per thread: 4 measured fastest for the decode workload (N=256, D=4096: 128 CTAs):
    // every CTA repeats the O(N) index check, so fewer, fuller CTAs cost less, and each
    // thread keeps four rows' loads in flight.  Fewer rows only when four would leave more
    // than half of the SMs idle.
    while (rows > 1 && 2 * gx * ((N + rl * rows - 1) / (rl * rows)) < static_cast<int64_t>(sms))
      rows /= 2;
    // A plain 4-row grid of more than one wave (one CTA per SM at its register count) runs
    // as 2-row CTAs instead, two to an SM.  Measured at S=512 W=4, us per step, 4 against 2
    // rows: D=4096 N=512 7.58 / 7.37, D=8192 N=256 7.43 / 6.96, D=8192 N=512 15.7 / 13.8.
    if (rows == 4 && mode == kUpdPlain && !off && gx * ((N + rl * 4 - 1) / (rl * 4)) > sms)
      rows = 2;
  }
#ifdef CCONV_TILE_SWEEP
  // Sweep builds only: CCONV_UPDATE_ROWS = 1, 2, 4, 8 or 16 forces the rows per thread.
  static const int rows_override = [] {
    const char* e = getenv("CCONV_UPDATE_ROWS");
    const int v = e ? atoi(e) : 0;
    return (v == 1 || v == 2 || v == 4 || v == 8 || v == 16) ? v : 0;
  }();
  if (rows_override) rows = rows_override;
#endif
  if (nt == kUpdThreadsSmall && rows > 4) rows = 4;
  if ((off || mode != kUpdPlain) && rows != 4) rows = 1;  // general kernels: 1 and 4 rows
  int64_t gy = (N + rl * rows - 1) / (rl * rows);
  // Row lanes: the kernel splits the N rows evenly over gridDim.y groups, each of at most
  // rl * rows rows as long as gy is at least the count above.  A grid short of the SM
  // count gets more, smaller groups, up to one CTA per SM (D=4096 N=256: 9 groups of 28-29
  // rows on 144 SMs instead of 8 of 32 on 128).
  bool balance = true;
#ifdef CCONV_TILE_SWEEP
  // Sweep builds only: CCONV_UPDATE_BALANCE=0 keeps the smallest row-group count.
  static const bool no_balance = [] {
    const char* e = getenv("CCONV_UPDATE_BALANCE");
    return e && atoi(e) == 0;
  }();
  balance = !no_balance;
#endif
  if (balance && rl > 1 && gx * gy < sms)
    gy = std::max(gy, std::min(static_cast<int64_t>(sms) / gx, N));
  if (gx > 2147483647 || gy > 65535) return CCONV_ERR_SHAPE;
  UpdKernel kern = vec8 ? (nt == kUpdThreadsSmall
                               ? pick_update_kernel<8, kUpdThreadsSmall>(W, rows, off, mode)
                               : pick_update_kernel<8, kUpdThreads>(W, rows, off, mode))
                        : pick_update_kernel<1, kUpdThreads>(W, rows, off, mode);
  if (!kern) return CCONV_ERR_SHAPE;

  UpdArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.state = static_cast<uint16_t*>(state);
  a.idx = state_indices;
  a.w = w;
  a.bias = bias;
  a.y = static_cast<uint16_t*>(y);
  a.status = status_dev;
  a.N = N;
  a.D = D;
  a.ldx = ldx;
  a.S = S;
  a.wdt = wdt;
  a.pad = pad ? 1 : 0;
  a.act = act;
  a.pos = pos;
  a.gq = N / gy;
  a.grem = N % gy;

  size_t smem = state_indices ? static_cast<size_t>((S + 31) / 32) * 4 : 0;
  if (rl > 1 && gx * gy <= sms) {
    // One CTA per SM.  The step is bound by each SM's load/store rate, and a grid of at most
    // one wave otherwise may be placed two CTAs to an SM (the 1- and 2-row kernels fit two)
    // with other SMs idle.  Dynamic shared memory of just over half an SM's capacity keeps
    // the CTAs apart.  Measured at S=512 W=4 (us per step, unpadded against padded):
    // D=4096 N=128 3.85 / 2.85, D=8192 N=64 3.70 / 2.79, D=2048 N=256 3.43 / 2.87.
    int per_sm = 0, reserved = 0;
    rc = smem_per_sm_current_device(&per_sm, &reserved);
    if (rc != CCONV_OK) return rc;
    const size_t half = static_cast<size_t>(per_sm / 2 - reserved + 16);
    if (half > smem) smem = half;
  }
#ifdef CCONV_TILE_SWEEP
  // Sweep builds only: CCONV_UPDATE_SMEM_PAD_KB pads the dynamic shared memory (caps the
  // CTAs that share an SM).
  static const size_t pad_kb = [] {
    const char* e = getenv("CCONV_UPDATE_SMEM_PAD_KB");
    const int v = e ? atoi(e) : 0;
    return static_cast<size_t>(v > 0 && v <= 200 ? v : 0);
  }();
  if (pad_kb * 1024 > smem) smem = pad_kb * 1024;
#endif
  // Dynamic plus static shared memory above 48 KB needs the per-function opt-in.
  if (smem > 32 * 1024) {
    if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)) != CCONV_OK)
      return CCONV_ERR_CUDA;
  }
  return launch_pdl(kern, dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                    dim3(nt), smem, reinterpret_cast<cudaStream_t>(stream), a) ==
                 cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}


}  // namespace cconv

extern "C" CCONV_API int cconv_update(const void* x, int64_t N, int64_t D, int64_t ldx,
                                      void* state, int64_t S, const int32_t* state_indices,
                                      const void* w, const void* bias, cconv_dtype wdt, int W,
                                      void* y, int32_t* status_dev, cconv_stream_t stream) {
  return cconv::update_impl(x, N, D, ldx, state, S, W - 1, state_indices, 0, nullptr, w, bias,
                            wdt, W, CCONV_ACT_SILU, y, status_dev, stream);
}

extern "C" CCONV_API int cconv_update_ex(const void* x, int64_t N, int64_t D, int64_t ldx,
                                         void* state, int64_t S, int L,
                                         const int32_t* state_indices, int pad_rows,
                                         const int32_t* cache_seqlens, const void* w,
                                         const void* bias, cconv_dtype wdt, int W,
                                         cconv_activation act, void* y, int32_t* status_dev,
                                         cconv_stream_t stream) {
  return cconv::update_impl(x, N, D, ldx, state, S, L, state_indices, pad_rows, cache_seqlens, w,
                            bias, wdt, W, act, y, status_dev, stream);
}
