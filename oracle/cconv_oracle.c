/*
 * cconv_oracle.c -- plain fp64 CPU statement of the depthwise causal short convolution
 * with fused SiLU: forward, backward and the single-token decode update.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle the CUDA path is checked against.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline / reference arm
 * may load it.  It shares no code, header, table or helper with the CUDA library, and the
 * library never calls it.
 *
 * Every function is written for a reader checking it against the definitions by eye:
 * straight loops in the order of the definition, fp64 arithmetic, libm exp(), no
 * blocking, no fusion, no reordering.  Sources (page title, file / section):
 *
 *   forward   y[b,t,d] = silu(bias[d] + sum_{k<W} w[d,W-1-k] * x[b,t-k,d]),
 *             x = 0 left of the sequence.
 *             kernel-fun 0.2.0.dev1 wheel, kernel_fun/cconv/_kernels/strip.py:
 *             `_tap` (w[:, W-1-k] multiplies x[t-k]), `_ld_ring` (zero left of the
 *             sequence), `_silu`.  The bias sits inside the activation (problem
 *             statement of the forward; the strip kernel itself carries no bias).
 *   backward  g = dy * s * (1 + z (1 - s)), s = sigmoid(z)    (strip.py `_dsilu`)
 *             dx[t] = sum_k w[d,W-1-k] * g[t+k], g = 0 past the end (strip.py `_bwd4`)
 *             dw[d,W-1-k] = sum_{b,t} g[t] * x[t-k]  (strip.py `_bwd4`, partial store
 *             at the end of `cconv_bwd_strip`), dbias[d] = sum_{b,t} g[b,t,d].
 *   decode    "Add experimental causal conv1d decode update - #797" (NVIDIA/cudnn-frontend),
 *             PR summary: per row i the state slot s = state_indices[i] is read, the new
 *             token emits y, then the state shifts by one and takes the token.  Negative,
 *             out-of-range and duplicate indices fail closed (nothing is mutated).
 *   packed    oracle_fwd_seq / oracle_bwd_seq: sequences packed along rows by cu_seqlens,
 *             an optional initial state per sequence, the final state a decode update
 *             continues from, and activation silu or none.  The keyword list fla's
 *             causal_conv1d takes (kernel-fun 0.2.0.dev1 wheel,
 *             kernel_fun/_common/compat.py: initial_state, output_final_state, activation,
 *             cu_seqlens), the follow-up scope and full-sequence-to-decode handoff of the
 *             cuDNN decode-update PR, and the decode state layout [.., D, W-1].
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - state[s,d,0] is the oldest entry; the window for the new token is
 *     (state[s,d,0..W-2], x[i,d]) and tap j multiplies window[j], which is the
 *     forward's orientation (window[W-1-k] = x[t-k]).
 *   - a repeated index is a "duplicate" only when it is in range; an out-of-range value
 *     is reported as out-of-range however often it occurs.
 *   - state_indices == NULL means row i uses slot i.
 *   - an initial state stands in for the W-1 rows before a sequence's first row, oldest
 *     first, the decode pool's layout; the final state is the last W-1 rows of the
 *     sequence extended by its initial state (or by zeros), so a sequence shorter than
 *     W-1 rows hands on part of its initial state.
 *
 * Number formats: the forward and backward take real values as double (the exact bf16
 * or fp32 values the GPU receives, widened by the caller), so they are plain functions of
 * real inputs.  The decode update moves state bits, so it takes the bf16 state and token
 * as their raw 16-bit patterns (uint16); a bf16 is the upper half of an IEEE-754
 * binary32, which is how it is widened for the arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_IDX_NEGATIVE 1
#define ORACLE_IDX_OUT_OF_RANGE 2
#define ORACLE_IDX_DUPLICATE 4

/* bf16 bit pattern -> double: the pattern is the top 16 bits of a binary32. */
static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

static double silu(double z) { return z * sigmoid(z); }

/* z[b,t,d] = bias[d] + sum_{k<W} w[d, W-1-k] * x[b, t-k, d], x[t-k] = 0 for t-k < 0 */
static double preactivation(int64_t T, int64_t D, int W, const double* x,
                            const double* w, const double* bias,
                            int64_t b, int64_t t, int64_t d) {
  double z = bias ? bias[d] : 0.0;
  for (int k = 0; k < W; ++k) {
    if (t - k < 0) continue;
    z += w[d * W + (W - 1 - k)] * x[(b * T + (t - k)) * D + d];
  }
  return z;
}

/* Forward. x: [B,T,D] contiguous.  w: [D,W].  bias: [D] or NULL.
 * y: [B,T,D] (fp64, unrounded).  z (optional, may be NULL): the pre-activation. */
int oracle_fwd(int64_t B, int64_t T, int64_t D, int W, const double* x,
               const double* w, const double* bias, double* y, double* z) {
  if (B < 0 || T < 0 || D < 0 || W < 1) return -1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double zz = preactivation(T, D, W, x, w, bias, b, t, d);
        if (z) z[(b * T + t) * D + d] = zz;
        y[(b * T + t) * D + d] = silu(zz);
      }
  return 0;
}

/* Backward. x, dy: [B,T,D] contiguous.  Outputs: dx [B,T,D], dw [D,W], dbias [D]
 * (dbias may be NULL).  z is recomputed from x, as the definition gives it. */
int oracle_bwd(int64_t B, int64_t T, int64_t D, int W, const double* x,
               const double* dy, const double* w, const double* bias,
               double* dx, double* dw, double* dbias) {
  if (B < 0 || T < 0 || D < 0 || W < 1) return -1;
  const int64_t n = B * T * D;
  double* g = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
  if (!g) return -2;

  /* g = dy * silu'(z),  silu'(z) = s (1 + z (1 - s)) */
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const int64_t i = (b * T + t) * D + d;
        const double zz = preactivation(T, D, W, x, w, bias, b, t, d);
        const double s = sigmoid(zz);
        g[i] = dy[i] * s * (1.0 + zz * (1.0 - s));
      }

  /* dx[b,t,d] = sum_{k<W} w[d, W-1-k] * g[b, t+k, d],  g = 0 for t+k >= T */
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int k = 0; k < W; ++k) {
          if (t + k >= T) continue;
          acc += w[d * W + (W - 1 - k)] * g[(b * T + (t + k)) * D + d];
        }
        dx[(b * T + t) * D + d] = acc;
      }

  /* dw[d, W-1-k] = sum_{b,t} g[b,t,d] * x[b,t-k,d] (x = 0 left of the sequence);
   * dbias[d] = sum_{b,t} g[b,t,d] */
  for (int64_t d = 0; d < D; ++d) {
    for (int j = 0; j < W; ++j) dw[d * W + j] = 0.0;
    if (dbias) dbias[d] = 0.0;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double gg = g[(b * T + t) * D + d];
        for (int k = 0; k < W; ++k) {
          if (t - k < 0) continue;
          dw[d * W + (W - 1 - k)] += gg * x[(b * T + (t - k)) * D + d];
        }
        if (dbias) dbias[d] += gg;
      }

  free(g);
  return 0;
}

/* ---------------------------------------------------------------------------------------
 * Packed sequences, initial / final state, activation.
 *
 * x holds nseq sequences packed along rows: sequence i is rows [cu[i], cu[i+1]) of the
 * [total, D] array (a batch of equal-length sequences is cu = 0, T, 2T, ...).  Inside each
 * sequence the convolution is the one above, except that the W-1 rows before its first row
 * come from init[i] when given (init[i][d][j] is row cu[i] - (W-1) + j, j = 0 the oldest)
 * and are zero otherwise.  act = 0: y = silu(z); act = 1: y = z (no activation).
 * final[i][d][j] (optional) is row cu[i+1] - (W-1) + j of that same extended sequence: the
 * state a decode update continues from.  The backward adds dinit[i][d][j] (optional), the
 * gradient of init[i][d][j]: sum_k w[d,W-1-k] g[u+k] over rows u+k inside the sequence,
 * u = cu[i] - (W-1) + j.  Readings: fla's causal_conv1d names initial_state /
 * output_final_state / cu_seqlens / activation (kernel-fun 0.2.0.dev1 wheel,
 * _common/compat.py); the decode update's state layout [.., D, W-1] fixes the state's shape.
 * --------------------------------------------------------------------------------------- */

/* value of sequence i's extended input at packed row u, channel d */
static double seq_x(int64_t D, int W, const double* x, const int64_t* cu, const double* init,
                    int64_t i, int64_t u, int64_t d) {
  if (u >= cu[i]) return x[u * D + d];
  const int64_t j = u - (cu[i] - (W - 1));
  if (j < 0 || !init) return 0.0;
  return init[(i * D + d) * (W - 1) + j];
}

/* pre-activation of sequence i at packed row t: bias + sum_k w[d, W-1-k] xe[t-k] */
static double seq_z(int64_t D, int W, const double* x, const int64_t* cu, const double* init,
                    const double* w, const double* bias, int64_t i, int64_t t, int64_t d) {
  double zs = bias ? bias[d] : 0.0;
  for (int k = 0; k < W; ++k) zs += w[d * W + (W - 1 - k)] * seq_x(D, W, x, cu, init, i, t - k, d);
  return zs;
}

int oracle_fwd_seq(int64_t nseq, const int64_t* cu, int64_t D, int W, const double* x,
                   const double* w, const double* bias, const double* init, int act,
                   double* y, double* final_state) {
  if (nseq < 0 || D < 0 || W < 1 || (act != 0 && act != 1)) return -1;
  for (int64_t i = 0; i < nseq; ++i) {
    if (cu[i + 1] < cu[i]) return -1;
    for (int64_t t = cu[i]; t < cu[i + 1]; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double zs = seq_z(D, W, x, cu, init, w, bias, i, t, d);
        y[t * D + d] = act == 0 ? silu(zs) : zs;
      }
    if (final_state)
      for (int64_t d = 0; d < D; ++d)
        for (int j = 0; j < W - 1; ++j)
          final_state[(i * D + d) * (W - 1) + j] =
              seq_x(D, W, x, cu, init, i, cu[i + 1] - (W - 1) + j, d);
  }
  return 0;
}

int oracle_bwd_seq(int64_t nseq, const int64_t* cu, int64_t D, int W, const double* x,
                   const double* dy, const double* w, const double* bias, const double* init,
                   int act, double* dx, double* dw, double* dbias, double* dinit) {
  if (nseq < 0 || D < 0 || W < 1 || (act != 0 && act != 1)) return -1;
  for (int64_t i = 0; i < nseq; ++i)
    if (cu[i + 1] < cu[i]) return -1;
  const int64_t total = nseq > 0 ? cu[nseq] : 0;
  double* gs = (double*)malloc((size_t)(total * D > 0 ? total * D : 1) * sizeof(double));
  if (!gs) return -2;
  /* gs = dy * act'(z) on every row of every sequence */
  for (int64_t i = 0; i < nseq; ++i)
    for (int64_t t = cu[i]; t < cu[i + 1]; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double gv = dy[t * D + d];
        if (act == 0) {
          const double zv = seq_z(D, W, x, cu, init, w, bias, i, t, d);
          const double sg = sigmoid(zv);
          gv *= sg * (1.0 + zv * (1.0 - sg));
        }
        gs[t * D + d] = gv;
      }
  for (int64_t d = 0; d < D; ++d) {
    for (int j = 0; j < W; ++j) dw[d * W + j] = 0.0;
    if (dbias) dbias[d] = 0.0;
  }
  for (int64_t i = 0; i < nseq; ++i) {
    const int64_t s = cu[i], e = cu[i + 1];
    /* dx[t] = sum_k w[d, W-1-k] gs[t+k], the sum stopping at the sequence's last row */
    for (int64_t t = s; t < e; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double ax = 0.0;
        for (int k = 0; k < W; ++k)
          if (t + k < e) ax += w[d * W + (W - 1 - k)] * gs[(t + k) * D + d];
        dx[t * D + d] = ax;
      }
    /* dw[d, W-1-k] += gs[t] xe[t-k]; dbias[d] += gs[t] (xe: the extended input) */
    for (int64_t t = s; t < e; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double gv = gs[t * D + d];
        for (int k = 0; k < W; ++k)
          dw[d * W + (W - 1 - k)] += gv * seq_x(D, W, x, cu, init, i, t - k, d);
        if (dbias) dbias[d] += gv;
      }
    /* gradient of the initial-state row u = s-(W-1)+j: the taps that reach into the
     * sequence from it */
    if (dinit)
      for (int64_t d = 0; d < D; ++d)
        for (int j = 0; j < W - 1; ++j) {
          const int64_t u = s - (W - 1) + j;
          double ai = 0.0;
          for (int k = 0; k < W; ++k)
            if (u + k >= s && u + k < e) ai += w[d * W + (W - 1 - k)] * gs[(u + k) * D + d];
          dinit[(i * D + d) * (W - 1) + j] = ai;
        }
  }
  free(gs);
  return 0;
}

/* Index validation for the decode update: bit mask of offences, 0 when every index is
 * in [0, S) and no in-range slot is named twice. */
int oracle_validate(int64_t N, int64_t S, const int32_t* idx) {
  int mask = 0;
  for (int64_t i = 0; i < N; ++i) {
    if (idx[i] < 0) mask |= ORACLE_IDX_NEGATIVE;
    else if (idx[i] >= S) mask |= ORACLE_IDX_OUT_OF_RANGE;
  }
  for (int64_t i = 0; i < N; ++i) {
    if (idx[i] < 0 || idx[i] >= S) continue;
    for (int64_t j = i + 1; j < N; ++j)
      if (idx[j] == idx[i]) mask |= ORACLE_IDX_DUPLICATE;
  }
  return mask;
}

/* Decode update.  x: [N,D] bf16 bits (contiguous).  state: [S,D,W-1] bf16 bits,
 * updated in place.  idx: [N] or NULL (row i -> slot i, needs S >= N).
 * w: [D,W], bias: [D] or NULL.  y: [N,D] fp64.
 * Returns 0, or the offence mask (> 0) with nothing written, or -1 on a bad shape. */
int oracle_update(int64_t N, int64_t D, int W, const uint16_t* x, uint16_t* state,
                  int64_t S, const int32_t* idx, const double* w, const double* bias,
                  double* y) {
  if (N < 0 || D < 0 || W < 1 || W > 8 || S < 0) return -1;
  if (idx) {
    const int mask = oracle_validate(N, S, idx);
    if (mask) return mask;
  } else if (S < N) {
    return -1;
  }
  const int L = W - 1; /* state length */
  uint16_t window[8];
  for (int64_t i = 0; i < N; ++i) {
    const int64_t s = idx ? (int64_t)idx[i] : i;
    if (s < 0 || s >= S) return -1; /* unreachable after a correct validation */
    for (int64_t d = 0; d < D; ++d) {
      uint16_t* st = state + (s * D + d) * L;
      for (int j = 0; j < L; ++j) window[j] = st[j];
      window[L] = x[i * D + d];
      double z = bias ? bias[d] : 0.0;
      for (int j = 0; j < W; ++j) z += w[d * W + j] * bf16_to_double(window[j]);
      y[i * D + d] = silu(z);
      for (int j = 0; j < L; ++j) st[j] = window[j + 1];
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------
 * Decode update, general form (the variants the cuDNN decode-update PR names): a state of
 * Ls >= W-1 entries per channel whose newest W-1 feed the window (Ls = W keeps one older
 * token); optional padding rows (pad != 0: an index of -1 marks a row that reads and writes
 * no state and produces no output -- its y row is left NaN here); activation silu (act = 0)
 * or none (act = 1).  Other negative, out-of-range or repeated indices fail closed as in
 * oracle_update.  Returns 0, the offence mask (> 0, nothing written), or -1 on a bad shape.
 * --------------------------------------------------------------------------------------- */
int oracle_validate_pad(int64_t N, int64_t S, const int32_t* idx, int pad) {
  int off = 0;
  for (int64_t i = 0; i < N; ++i) {
    const int32_t v = idx[i];
    if (pad && v == -1) continue; /* a padding row */
    if (v < 0) off |= ORACLE_IDX_NEGATIVE;
    else if (v >= S) off |= ORACLE_IDX_OUT_OF_RANGE;
    else
      for (int64_t k = 0; k < i; ++k)
        if (idx[k] == v) off |= ORACLE_IDX_DUPLICATE;
  }
  return off;
}

int oracle_update_ex(int64_t N, int64_t D, int W, int Ls, const uint16_t* x, uint16_t* state,
                     int64_t S, const int32_t* idx, int pad, const double* w, const double* bias,
                     int act, double* y) {
  if (N < 0 || D < 0 || W < 1 || W > 8 || Ls < W - 1 || Ls > 8 || S < 0) return -1;
  if (act != 0 && act != 1) return -1;
  if (idx) {
    const int off = oracle_validate_pad(N, S, idx, pad);
    if (off) return off;
  } else if (S < N) {
    return -1;
  }
  uint16_t win[8];
  for (int64_t i = 0; i < N; ++i) {
    const int64_t slot = idx ? (int64_t)idx[i] : i;
    if (idx && pad && idx[i] == -1) {
      for (int64_t d = 0; d < D; ++d) y[i * D + d] = NAN;
      continue;
    }
    if (slot < 0 || slot >= S) return -1; /* unreachable after a correct validation */
    for (int64_t d = 0; d < D; ++d) {
      uint16_t* cell = state + (slot * D + d) * Ls;
      /* window: the newest W-1 state entries, then the token */
      for (int j = 0; j < W - 1; ++j) win[j] = cell[Ls - (W - 1) + j];
      win[W - 1] = x[i * D + d];
      double zd = bias ? bias[d] : 0.0;
      for (int j = 0; j < W; ++j) zd += w[d * W + j] * bf16_to_double(win[j]);
      y[i * D + d] = act == 0 ? silu(zd) : zd;
      /* the state drops its oldest entry and takes the token */
      for (int j = 0; j + 1 < Ls; ++j) cell[j] = cell[j + 1];
      if (Ls > 0) cell[Ls - 1] = x[i * D + d];
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------
 * Decode update, circular-buffer form (the cache_seqlens mode the cuDNN decode-update PR
 * reserves).  Reading: the state of a slot is a ring of Ls >= W-1 entries per channel, and
 * pos[i] counts the tokens slot s has already seen.  The new token goes to ring entry
 * pos[i] mod Ls (taken non-negative); the window is the W-1 ring entries before it
 * (positions pos-(W-1) .. pos-1 mod Ls, oldest first), then the token.  Nothing is shifted;
 * the caller advances pos.  Padding rows, activation and validation as oracle_update_ex.
 * --------------------------------------------------------------------------------------- */
static int64_t ring_mod(int64_t a, int64_t m) {
  const int64_t r = a % m;
  return r < 0 ? r + m : r;
}

int oracle_update_ring(int64_t N, int64_t D, int W, int Ls, const uint16_t* x, uint16_t* state,
                       int64_t S, const int32_t* idx, int pad, const int32_t* pos,
                       const double* w, const double* bias, int act, double* y) {
  if (N < 0 || D < 0 || W < 1 || W > 8 || Ls < W - 1 || Ls < 1 || Ls > 8 || S < 0) return -1;
  if (act != 0 && act != 1) return -1;
  if (idx) {
    const int off = oracle_validate_pad(N, S, idx, pad);
    if (off) return off;
  } else if (S < N) {
    return -1;
  }
  uint16_t ring_win[8];
  for (int64_t i = 0; i < N; ++i) {
    if (pad && idx && idx[i] == -1) { /* a padding row: no state access, no output */
      for (int64_t d = 0; d < D; ++d) y[i * D + d] = NAN;
      continue;
    }
    const int64_t slot = idx ? (int64_t)idx[i] : i;
    if (slot < 0 || slot >= S) return -1;
    const int64_t head = ring_mod(pos[i], Ls); /* where the new token goes */
    for (int64_t d = 0; d < D; ++d) {
      uint16_t* ring = state + (slot * D + d) * Ls;
      for (int j = 0; j < W - 1; ++j) ring_win[j] = ring[ring_mod(head - (W - 1) + j, Ls)];
      ring_win[W - 1] = x[i * D + d];
      double zr = bias ? bias[d] : 0.0;
      for (int j = 0; j < W; ++j) zr += w[d * W + j] * bf16_to_double(ring_win[j]);
      y[i * D + d] = act == 0 ? silu(zr) : zr;
      ring[head] = x[i * D + d];
    }
  }
  return 0;
}
