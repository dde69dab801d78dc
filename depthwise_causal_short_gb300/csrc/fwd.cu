// fwd.cu -- cconv_fwd: the forward stream (one kernel).
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
  uint16_t* y;  // [B,T,D] contiguous bf16
  int64_t D;
  int T, BT;
  int cpc;      // CTAs per channel group
  int W, wdt;
};

// One output row from the new input row x and the ring h = (x[t-1], x[t-2], x[t-3]).
// With halved taps hz = z / 2, and silu(z) = hz * (1 + tanh(hz)).
template <int P>
__device__ __forceinline__ void fwd_row(const f2 (&x)[P], const f2 (&h)[3][P],
                                        const f2 (&tap)[4][P], const f2 (&bias2)[P],
                                        f2 (&yv)[P]) {
#pragma unroll
  for (int q = 0; q < P; ++q) {
    f2 hz = f2_fma(tap[0][q], x[q], bias2[q]);
    hz = f2_fma(tap[1][q], h[0][q], hz);
    hz = f2_fma(tap[2][q], h[1][q], hz);
    hz = f2_fma(tap[3][q], h[2][q], hz);
    yv[q] = f2_fma(hz, f2_tanh(hz), hz);
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
template <int VEC, int R, bool FULL, bool STORE>
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
        fwd_row<P>(x, h, tap, bias2, yv);
        if (STORE || active) store_row<VEC>(yrow, yv);
      }
      ring_push<P>(h, x);
    }
    yrow += p.D;
  }
}

// Loads one tile (rows cur.tt .. cur.tt+R-1, one box per consumer warp) into a stage.
template <int VEC, int R, int NC>
__device__ __forceinline__ void fwd_issue(uint8_t* st, uint64_t* full, const CUtensorMap* tmx,
                                          const TileCursor& cur, int nact, int c0, uint64_t pol) {
  constexpr int CB = 32 * VEC;
  constexpr int TILE = R * CB * 2;
  mbar_arrive_expect_tx(full, nact * TILE);
  for (int w = 0; w < nact; ++w)
    tma_load_3d(st + w * TILE, tmx, full, c0 + w * CB, cur.tt, cur.b, pol);
}

// CTA: NC consumer warps (warp w owns channels c0 + w*CB .. c0 + (w+1)*CB - 1 of every tile).
// SEP: a separate producer warp (index NC) streams the stages; otherwise lane 0 of consumer
// warp 0 re-arms each stage once every consumer has released it.  Stage layout: NC boxes of
// R rows x CB channels.
template <int VEC, int R, int S, int NC, int MINB, bool SEP>
__global__ void __maxnreg__(regs_for(NC + SEP, MINB))
cconv_fwd_kernel(const __grid_constant__ CUtensorMap tmx, const FwdArgs p) {
  constexpr int CB = 32 * VEC;
  constexpr int TILE = R * CB * 2;
  constexpr int STAGE = NC * TILE;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
  uint64_t* empty = full + S;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cg = blockIdx.x / p.cpc;
  const int part = blockIdx.x - cg * p.cpc;
  const int r0 = static_cast<int>(static_cast<int64_t>(part) * p.BT / p.cpc);
  const int r1 = static_cast<int>(static_cast<int64_t>(part + 1) * p.BT / p.cpc);
  const int c0 = cg * NC * CB;
  int nact = static_cast<int>((p.D - c0 + CB - 1) / CB);  // consumer warps with channels
  if (nact > NC) nact = NC;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmx);
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

  TileCursor cur;
  cur.init(r0, r1, p.T, 0, R);
  const uint64_t pol = policy_evict_first();
  if (SEP && warp == NC) {
    // ---- producer warp -------------------------------------------------------------------
    if (lane == 0) {
      uint32_t eph = 0;
      int s = 0;
      for (int i = 0; !cur.done; ++i) {
        if (i >= S) {  // wait until every consumer has released this stage
          if (!mbar_wait_bounded(&empty[s], (eph >> s) & 1u, kWaitLimitNs)) {
            atomicOr(&g_fault_fwd, kFaultFwdWait);
            break;
          }
          eph ^= 1u << s;
        }
        fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], &tmx, cur, nact, c0, pol);
        cur.advance();
        s = (s + 1 == S) ? 0 : s + 1;
      }
    }
  } else if (warp < nact) {
    // ---- consumer ------------------------------------------------------------------------
    const bool leader = !SEP && warp == 0;
    TileCursor pc = cur;  // the leader's producer cursor, S tiles ahead
    if (leader && lane == 0) {
      for (int s = 0; s < S && !pc.done; ++s) {
        fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], &tmx, pc, nact, c0, pol);
        pc.advance();
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
      if (cur.from == cur.tt && cur.tt >= cur.a && cur.tt + R <= cur.e) {
        if (all_active)
          fwd_tile<VEC, R, true, true>(tile, lane, cur, active, p, d0, tap, bias2, h);
        else
          fwd_tile<VEC, R, true, false>(tile, lane, cur, active, p, d0, tap, bias2, h);
      } else {
        fwd_tile<VEC, R, false, false>(tile, lane, cur, active, p, d0, tap, bias2, h);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (leader) {
        // Re-arm this stage with the tile S ahead once every consumer has released it.
        bool fine = true;
        if (lane == 0 && !pc.done) {
          fine = mbar_wait_bounded(&empty[s], (eph >> s) & 1u, kWaitLimitNs);
          if (fine) {
            fwd_issue<VEC, R, NC>(smem + s * STAGE, &full[s], &tmx, pc, nact, c0, pol);
            pc.advance();
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
  }
  grid_launch_dependents();
}

// ------------------------------------------------------------------------------------
// launch configurations (compile-time tile shapes; the first is the default)
// ------------------------------------------------------------------------------------
struct FwdConfig {
  int vec, rows, stages, nc, ctas_per_sm, sep;
  void (*kernel)(const CUtensorMap, const FwdArgs);
};

#define CCONV_FWD_CFG(V, R, S, NC, M, SEP) \
  FwdConfig { V, R, S, NC, M, SEP, cconv_fwd_kernel<V, R, S, NC, M, SEP> }

static const FwdConfig kFwdConfigs[] = {
    CCONV_FWD_CFG(4, 8, 10, 8, 1, true),  // measured fastest at B=2 T=8192 D=4096
    CCONV_FWD_CFG(4, 12, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 16, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 24, 4, 8, 1, true),
    CCONV_FWD_CFG(4, 12, 4, 8, 2, true),
    CCONV_FWD_CFG(8, 8, 6, 8, 1, true),
    CCONV_FWD_CFG(4, 8, 5, 8, 2, false),
    CCONV_FWD_CFG(4, 4, 20, 8, 1, true),
};
static const int kNumFwdConfigs = sizeof(kFwdConfigs) / sizeof(kFwdConfigs[0]);

static int fwd_config_index() {
  static int idx = -1;
  if (idx < 0) {
    const char* e = getenv("CCONV_FWD_CONFIG");
    int v = e ? atoi(e) : 0;
    idx = (v >= 0 && v < kNumFwdConfigs) ? v : 0;
  }
  return idx;
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
