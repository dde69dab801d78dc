// fwd.cu -- cconv_fwd: the forward stream (one kernel).
//
// y[b,t,d] = silu(bias[d] + sum_{k<W} w[d,W-1-k] * x[b,t-k,d]), x = 0 left of the sequence.
// Definition: kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py (`_tap`,
// `_ld_ring`, `_silu`, `_fwd4`); its module docstring gives the design point this kernel
// keeps: one load of x, one sigmoid and one store per element, the W-1 previous rows held
// in registers.
//
// What differs from that Triton design: x does not travel through registers on its way in.
// Each warp runs its own TMA pipeline: its lane 0 keeps S tiles of R rows x (32*VEC)
// channels in flight into shared memory, each completing on an mbarrier, so the bytes in
// flight per SM are set by shared memory (S * tile bytes per warp) rather than by the
// register budget, which was the limit the pages measured.  The 3 ring rows before a range
// and the zero padding before t = 0 come from the same tiled copy (out-of-range rows fill
// with zeros).  Arithmetic is packed f32x2; the sigmoid is 0.5 * tanh.approx(z/2) + 0.5.
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
  int n_cb, wpc, total_warps;
  int W, wdt;
};

template <int VEC, int R>
__device__ __forceinline__ void fwd_tile(const uint8_t* tile, int lane, const TileCursor& c,
                                         bool full, bool active, const FwdArgs& p, int64_t d0,
                                         const f2 (&tap)[4][VEC / 2], const f2 (&bias2)[VEC / 2],
                                         f2 (&h)[3][VEC / 2]) {
  constexpr int P = VEC / 2;
  constexpr int ROWB = 32 * VEC * 2;
  uint16_t* ybase = p.y + static_cast<int64_t>(c.b) * p.T * p.D + d0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int t = c.tt + i;
    if (!full && t < c.from) continue;  // processed with the previous tile
    f2 x[P];
    smem_row<VEC>(tile + i * ROWB, lane, x);
    const bool emit = full || (t >= c.a && t < c.e);
    if (emit) {
      f2 yv[P];
#pragma unroll
      for (int q = 0; q < P; ++q) {
        f2 z = f2_fma(tap[0][q], x[q], bias2[q]);
        z = f2_fma(tap[1][q], h[0][q], z);
        z = f2_fma(tap[2][q], h[1][q], z);
        z = f2_fma(tap[3][q], h[2][q], z);
        yv[q] = f2_silu(z);
      }
      if (active) store_row<VEC>(ybase + static_cast<int64_t>(t) * p.D, yv);
    }
#pragma unroll
    for (int q = 0; q < P; ++q) {
      h[2][q] = h[1][q];
      h[1][q] = h[0][q];
      h[0][q] = x[q];
    }
  }
}

template <int VEC, int R, int S, int NW>
__global__ void __launch_bounds__(NW * 32, 1)
cconv_fwd_kernel(const __grid_constant__ CUtensorMap tmx, const FwdArgs p) {
  constexpr int CB = 32 * VEC;
  constexpr int TILE = R * CB * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * NW + warp;
  if (gw >= p.total_warps) {  // no CTA-wide barrier follows
    grid_launch_dependents();
    return;
  }

  uint8_t* tiles = smem + warp * (S * TILE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * S * TILE) + warp * S;

  // Strips vary fastest along the warp index, so the warps of a CTA read neighbouring
  // strips of the same rows at about the same time (contiguous row segments in DRAM).
  const int k = gw / p.n_cb;
  const int cb = gw - k * p.n_cb;
  const int r0 = static_cast<int>(static_cast<int64_t>(k) * p.BT / p.wpc);
  const int r1 = static_cast<int>(static_cast<int64_t>(k + 1) * p.BT / p.wpc);
  const int c0 = cb * CB;
  const int64_t d0 = c0 + lane * VEC;
  const bool active = d0 < p.D;

  if (lane == 0) {
    prefetch_tensormap(&tmx);
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Everything above touches no global memory; from here on the previous kernel on the
  // stream has completed.
  grid_dependency_wait();

  TileCursor pc, cc;
  pc.init(r0, r1, p.T, 0, R);
  cc = pc;
  const uint64_t pol = policy_evict_first();
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      if (!pc.done) {
        mbar_arrive_expect_tx(&bars[s], TILE);
        tma_load_3d(tiles + s * TILE, &tmx, &bars[s], c0, pc.tt, pc.b, pol);
        pc.advance();
      }
    }
  }

  // Taps load while the first tiles are in flight.
  f2 tap[4][VEC / 2], bias2[VEC / 2];
  load_taps<VEC>(p.w, p.bias, p.wdt, p.W, d0, active, tap, bias2);

  f2 h[3][VEC / 2];
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int q = 0; q < VEC / 2; ++q) h[j][q] = 0ull;

  uint32_t parity = 0;  // bit s: phase parity expected next on stage s
  int s = 0;
  while (!cc.done) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[s], (parity >> s) & 1u,
                                                             kWaitLimitNs));
    if (!ok) {
      if (lane == 0) atomicOr(&g_fault_fwd, kFaultFwdWait);
      // Let this warp's other copies land (bounded) before the CTA can exit.
      for (int j = 0; j < S; ++j) (void)mbar_wait_bounded(&bars[j], (parity >> j) & 1u, 100000000ull);
      return;
    }
    parity ^= 1u << s;
    const uint8_t* tile = tiles + s * TILE;
    const bool full = cc.from == cc.tt && cc.tt >= cc.a && cc.tt + R <= cc.e;
    if (full)
      fwd_tile<VEC, R>(tile, lane, cc, true, active, p, d0, tap, bias2, h);
    else
      fwd_tile<VEC, R>(tile, lane, cc, false, active, p, d0, tap, bias2, h);
    __syncwarp();
    if (lane == 0 && !pc.done) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bars[s], TILE);
      tma_load_3d(tiles + s * TILE, &tmx, &bars[s], c0, pc.tt, pc.b, pol);
      pc.advance();
    }
    cc.advance();
    s = (s + 1 == S) ? 0 : s + 1;
  }
  grid_launch_dependents();
}

// ------------------------------------------------------------------------------------
// launch configurations (compile-time tile shapes; the first is the default)
// ------------------------------------------------------------------------------------
struct FwdConfig {
  int vec, rows, stages, warps;
  void (*kernel)(const CUtensorMap, const FwdArgs);
};

#define CCONV_FWD_CFG(V, R, S, NW) \
  FwdConfig { V, R, S, NW, cconv_fwd_kernel<V, R, S, NW> }

static const FwdConfig kFwdConfigs[] = {
    CCONV_FWD_CFG(4, 16, 4, 8),  // measured fastest at B=2 T=8192 D=4096
    CCONV_FWD_CFG(8, 8, 4, 8),
    CCONV_FWD_CFG(8, 16, 3, 8),
    CCONV_FWD_CFG(8, 16, 4, 4),
    CCONV_FWD_CFG(8, 8, 3, 16),
    CCONV_FWD_CFG(4, 16, 3, 16),
    CCONV_FWD_CFG(4, 8, 4, 16),
    CCONV_FWD_CFG(8, 8, 2, 16),
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
  const StripPlan plan = make_strip_plan(B, T, D, cfg.vec, cfg.warps, 1, sms, 32);

  normalise_strides(B, T, D, sxb, sxt);
  CUtensorMap tmx;
  rc = encode_rows_map(&tmx, x, B, T, D, sxb, sxt, 32 * cfg.vec, cfg.rows);
  if (rc != CCONV_OK) return rc;

  FwdArgs a;
  a.w = w;
  a.bias = bias;
  a.y = static_cast<uint16_t*>(y);
  a.T = static_cast<int>(T);
  a.D = D;
  a.BT = static_cast<int>(B * T);
  a.n_cb = plan.n_cb;
  a.wpc = plan.wpc;
  a.total_warps = plan.total_warps;
  a.W = W;
  a.wdt = wdt;

  const int smem = cfg.warps * cfg.stages * (cfg.rows * 32 * cfg.vec * 2 + 8);
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(cfg.kernel), smem);
  if (rc != CCONV_OK) return rc;
  return launch_pdl(cfg.kernel, dim3(plan.grid), dim3(cfg.warps * 32), smem,
                    reinterpret_cast<cudaStream_t>(stream), tmx, a) == cudaSuccess
             ? CCONV_OK
             : CCONV_ERR_CUDA;
}
