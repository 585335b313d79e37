/*
 * CPU oracle for the TwELL activation-sparse feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library; the product path never does.  It shares
 * no code, header or table with the CUDA library.
 *
 * What it computes follows "Sparser, Faster, Lighter Transformer Language
 * Models" (Sakana AI + NVIDIA) as described on the pages:
 *   - the FFN nonlinearity is a ReLU whose zeros are the sparsity
 *     (iaexpertos blog, "The Challenge of Sparsity Ignored by GPUs");
 *   - TwELL = Tile-wise ELLPACK (ifai.io news, "Reshaping math for the GPU";
 *     repo-explainer, "TwELL: The Packing Format That Fits the Machine");
 *   - storage is three arrays: non-zero values, tile-local indices, per-tile
 *     non-zero counts, with tile size T and tile index t (bayesiansapien note,
 *     flowchart and the description of the paper's Figure 1);
 *   - a hybrid splits rows between TwELL and a dense matrix that catches the
 *     rare dense tokens (ifai.io news, "Reshaping math for the GPU"; Figure 1
 *     "hybrid" in the bayesiansapien note);
 *   - L1 regularisation of the activations induces the sparsity and its
 *     gradient belongs to training (bayesiansapien note, TL;DR).
 *
 * Precision: inputs are bf16 bit patterns (uint16).  Every dot product is a
 * plain fp32 loop with the summation index ascending (the layer specification
 * asks for fp32 accumulation).  Rounding to bf16 is round-to-nearest-even,
 * written from the IEEE-754 definition.  Compile with -ffp-contract=off so that
 * no multiply-add is fused and results agree across hosts.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   capacity C per (row, tile); a row with any tile count > C goes whole to the
 *   dense fallback; layout [row][tile][slot]; u8 indices and counts; padding
 *   value +0.0 and index 0; entries in ascending tile-local index; fallback
 *   slots in ascending row order; non-zero means bf16(h) != 0 after rounding;
 *   bias added in fp32 before the ReLU; no down-projection bias; the L1 term is
 *   lambda * sum |h| so its gradient is lambda wherever h > 0.
 *   The tile-granular hybrid (a variant the pages do not spell out) keeps an
 *   over-full tile densely in a pool, slots in (row, tile) order, the slot
 *   number in the cell's first entry and the count set to 255.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

static float bf16_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round to nearest, ties to even, on the 16 bits that bf16 keeps.  Finite
 * inputs only (the generator never produces NaN or Inf). */
static uint16_t f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  uint32_t keep = u >> 16;
  uint32_t rest = u & 0xFFFFu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

EXPORT uint16_t oracle_bf16_round(float x) { return f32_to_bf16(x); }

/* z[r][j] = sum_k X[row][k] * W_inT[j][k] (k ascending) + b[j];
 * h = bf16(z) if z > 0 else +0.  Rows are taken from the list `rows`. */
EXPORT void oracle_hidden(const uint16_t* X, const uint16_t* W_inT, const uint16_t* b,
                          int32_t d, int32_t f, const int32_t* rows, int32_t n_sel,
                          float* Z, uint16_t* H) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    const uint16_t* x = X + (int64_t)rows[r] * d;
    for (int32_t j = 0; j < f; ++j) {
      const uint16_t* w = W_inT + (int64_t)j * d;
      float acc = 0.0f;
      for (int32_t k = 0; k < d; ++k) acc += bf16_to_f32(x[k]) * bf16_to_f32(w[k]);
      float z = acc + bf16_to_f32(b[j]);
      if (Z) Z[(int64_t)r * f + j] = z;
      if (H) H[(int64_t)r * f + j] = (z > 0.0f) ? f32_to_bf16(z) : (uint16_t)0;
    }
  }
}

/* Gated variant: h = bf16(zg * zu) where zg > 0 else +0, zg carrying the bias. */
EXPORT void oracle_hidden_gated(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                const uint16_t* b, int32_t d, int32_t f, const int32_t* rows,
                                int32_t n_sel, float* Zg, uint16_t* H) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    const uint16_t* x = X + (int64_t)rows[r] * d;
    for (int32_t j = 0; j < f; ++j) {
      const uint16_t* wg = W_gT + (int64_t)j * d;
      const uint16_t* wu = W_uT + (int64_t)j * d;
      float g = 0.0f, u = 0.0f;
      for (int32_t k = 0; k < d; ++k) {
        g += bf16_to_f32(x[k]) * bf16_to_f32(wg[k]);
        u += bf16_to_f32(x[k]) * bf16_to_f32(wu[k]);
      }
      g += bf16_to_f32(b[j]);
      if (Zg) Zg[(int64_t)r * f + j] = g;
      if (H) H[(int64_t)r * f + j] = (g > 0.0f) ? f32_to_bf16(g * u) : (uint16_t)0;
    }
  }
}

/* Scalar-loop TwELL packer.  For each row and tile, walk the tile's T columns
 * in ascending order; every non-zero increments the tile's count and, while
 * the count is <= C, is stored in the next slot with its tile-local index.
 * A row with any tile count above C goes to the dense fallback: fallback rows
 * get slots in ascending row order, their dense row is copied to fb_dense, and
 * their TwELL counts and slots stay zero.  Returns the number of fallback rows
 * (which may exceed fb_cap; rows past the capacity are not stored). */
EXPORT int32_t oracle_pack(const uint16_t* H, int32_t N, int32_t f, int32_t T, int32_t C,
                           int32_t fb_cap, uint16_t* values, uint8_t* idx, uint8_t* counts,
                           int32_t* row_fb, int32_t* fb_rows, uint16_t* fb_dense) {
  const int32_t nt = f / T;
  int32_t n_fb = 0;
  for (int32_t n = 0; n < N; ++n) {
    const uint16_t* h = H + (int64_t)n * f;
    int overflow = 0;
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      int32_t cnt = 0;
      for (int32_t s = 0; s < C; ++s) {
        values[cell * C + s] = 0;
        idx[cell * C + s] = 0;
      }
      for (int32_t i = 0; i < T; ++i) {
        uint16_t v = h[(int64_t)t * T + i];
        if (bf16_to_f32(v) != 0.0f) {
          cnt += 1;
          if (cnt <= C) {
            values[cell * C + cnt - 1] = v;
            idx[cell * C + cnt - 1] = (uint8_t)i;
          }
        }
      }
      if (cnt > C) overflow = 1;
      counts[cell] = (uint8_t)(cnt > C ? C : cnt);
    }
    if (overflow) {
      for (int32_t t = 0; t < nt; ++t) {
        int64_t cell = (int64_t)n * nt + t;
        counts[cell] = 0;
        for (int32_t s = 0; s < C; ++s) {
          values[cell * C + s] = 0;
          idx[cell * C + s] = 0;
        }
      }
      row_fb[n] = n_fb;
      if (n_fb < fb_cap) {
        fb_rows[n_fb] = n;
        memcpy(fb_dense + (int64_t)n_fb * f, h, sizeof(uint16_t) * (size_t)f);
      }
      n_fb += 1;
    } else {
      row_fb[n] = -1;
    }
  }
  return n_fb;
}

/* TwELL -> dense: zero H, write each stored value at column t*T + idx; copy
 * fallback rows from fb_dense. */
EXPORT void oracle_unpack(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                          const int32_t* row_fb, const uint16_t* fb_dense, int32_t N, int32_t f,
                          int32_t T, int32_t C, int32_t fb_cap, uint16_t* H) {
  const int32_t nt = f / T;
  for (int32_t n = 0; n < N; ++n) {
    uint16_t* h = H + (int64_t)n * f;
    if (row_fb[n] >= 0) {
      /* a fallback row past the capacity is stored nowhere (its cells are
       * empty too): it comes back as zeros */
      if (row_fb[n] < fb_cap)
        memcpy(h, fb_dense + (int64_t)row_fb[n] * f, sizeof(uint16_t) * (size_t)f);
      else
        memset(h, 0, sizeof(uint16_t) * (size_t)f);
      continue;
    }
    memset(h, 0, sizeof(uint16_t) * (size_t)f);
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      for (int32_t s = 0; s < counts[cell]; ++s) h[(int64_t)t * T + idx[cell * C + s]] = values[cell * C + s];
    }
  }
}

/* Tile-granular hybrid (a variant of the paper's Figure 1 as the bayesiansapien
 * note describes it: the hybrid splits between TwELL and a dense store; here
 * the unit of the split is one (row, tile) cell instead of a whole row).  A
 * tile whose non-zero count exceeds C is kept densely: its T values go to the
 * next slot of the tile pool (slots numbered in ascending (row, tile) order),
 * the cell's count is 255 and the slot number sits in the cell's first entry
 * (value = low 16 bits, index = bits 16..23; the other C - 1 slots are
 * padding).  Tiles with at most C non-zeros are packed as in oracle_pack.  No
 * row is routed whole: row_fb is -1 everywhere.  Returns the number of dense
 * tiles, which may exceed pool_cap; dense tiles past the capacity are not
 * stored and their cells stay empty (count 0).  Needs C >= 1. */
EXPORT int32_t oracle_pack_tiles(const uint16_t* H, int32_t N, int32_t f, int32_t T, int32_t C, int32_t pool_cap,
                                 uint16_t* values, uint8_t* idx, uint8_t* counts, int32_t* row_fb,
                                 uint16_t* pool) {
  const int32_t nt = f / T;
  int32_t n_dense = 0;
  for (int32_t n = 0; n < N; ++n) {
    const uint16_t* h = H + (int64_t)n * f;
    row_fb[n] = -1;
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      int32_t cnt = 0;
      for (int32_t s = 0; s < C; ++s) {
        values[cell * C + s] = 0;
        idx[cell * C + s] = 0;
      }
      for (int32_t i = 0; i < T; ++i) {
        uint16_t v = h[(int64_t)t * T + i];
        if (bf16_to_f32(v) != 0.0f) {
          if (cnt < C) {
            values[cell * C + cnt] = v;
            idx[cell * C + cnt] = (uint8_t)i;
          }
          cnt += 1;
        }
      }
      if (cnt > C) {
        /* dense tile: the entries written above become padding again */
        for (int32_t s = 0; s < C; ++s) {
          values[cell * C + s] = 0;
          idx[cell * C + s] = 0;
        }
      } else {
        counts[cell] = (uint8_t)cnt;
        continue;
      }
      if (n_dense < pool_cap) {
        counts[cell] = 255;
        values[cell * C] = (uint16_t)(n_dense & 0xFFFF);
        idx[cell * C] = (uint8_t)((n_dense >> 16) & 0xFF);
        memcpy(pool + (int64_t)n_dense * T, h + (int64_t)t * T, sizeof(uint16_t) * (size_t)T);
      } else {
        counts[cell] = 0;
      }
      n_dense += 1;
    }
  }
  return n_dense;
}

/* Tile-granular hybrid -> dense: zero H, write the stored entries, copy each
 * dense tile from its pool slot. */
EXPORT void oracle_unpack_tiles(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                                const uint16_t* pool, int32_t N, int32_t f, int32_t T, int32_t C, uint16_t* H) {
  const int32_t nt = f / T;
  for (int32_t n = 0; n < N; ++n) {
    uint16_t* h = H + (int64_t)n * f;
    memset(h, 0, sizeof(uint16_t) * (size_t)f);
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      if (counts[cell] == 255) {
        int64_t slot = (int64_t)values[cell * C] | ((int64_t)idx[cell * C] << 16);
        memcpy(h + (int64_t)t * T, pool + slot * T, sizeof(uint16_t) * (size_t)T);
        continue;
      }
      for (int32_t s = 0; s < counts[cell]; ++s) h[(int64_t)t * T + idx[cell * C + s]] = values[cell * C + s];
    }
  }
}

/* Y from the tile-granular hybrid: stored entries of each tile, or the dense
 * tile's non-zeros walked in column order, so j ascends as in oracle_down_dense. */
EXPORT void oracle_down_packed_tiles(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                                     const uint16_t* pool, const uint16_t* W_down, int32_t N, int32_t f, int32_t d,
                                     int32_t T, int32_t C, float* Y) {
  const int32_t nt = f / T;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t n = 0; n < N; ++n) {
    float* y = Y + (int64_t)n * d;
    for (int32_t c = 0; c < d; ++c) {
      float acc = 0.0f;
      for (int32_t t = 0; t < nt; ++t) {
        int64_t cell = (int64_t)n * nt + t;
        if (counts[cell] == 255) {
          const uint16_t* tile = pool + ((int64_t)values[cell * C] | ((int64_t)idx[cell * C] << 16)) * T;
          for (int32_t i = 0; i < T; ++i)
            if (bf16_to_f32(tile[i]) != 0.0f)
              acc += bf16_to_f32(tile[i]) * bf16_to_f32(W_down[((int64_t)t * T + i) * d + c]);
          continue;
        }
        for (int32_t s = 0; s < counts[cell]; ++s) {
          int32_t j = t * T + idx[cell * C + s];
          acc += bf16_to_f32(values[cell * C + s]) * bf16_to_f32(W_down[(int64_t)j * d + c]);
        }
      }
      y[c] = acc;
    }
  }
}

/* Y[r][c] = sum_j H[r][j] * W_down[j][c], j ascending, fp32. */
EXPORT void oracle_down_dense(const uint16_t* H, const uint16_t* W_down, int32_t n_sel, int32_t f,
                              int32_t d, float* Y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    const uint16_t* h = H + (int64_t)r * f;
    float* y = Y + (int64_t)r * d;
    for (int32_t c = 0; c < d; ++c) {
      float acc = 0.0f;
      for (int32_t j = 0; j < f; ++j) acc += bf16_to_f32(h[j]) * bf16_to_f32(W_down[(int64_t)j * d + c]);
      y[c] = acc;
    }
  }
}

/* The same product read from the packed form: TwELL rows visit their stored
 * entries tile by tile (so j ascends), fallback rows walk their dense row. */
EXPORT void oracle_down_packed(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                               const int32_t* row_fb, const uint16_t* fb_dense,
                               const uint16_t* W_down, int32_t N, int32_t f, int32_t d, int32_t T,
                               int32_t C, int32_t fb_cap, float* Y) {
  const int32_t nt = f / T;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t n = 0; n < N; ++n) {
    float* y = Y + (int64_t)n * d;
    for (int32_t c = 0; c < d; ++c) {
      float acc = 0.0f;
      if (row_fb[n] >= 0) {
        /* a fallback row past the capacity is stored nowhere: a zero row */
        if (row_fb[n] < fb_cap) {
          const uint16_t* h = fb_dense + (int64_t)row_fb[n] * f;
          for (int32_t j = 0; j < f; ++j)
            if (bf16_to_f32(h[j]) != 0.0f) acc += bf16_to_f32(h[j]) * bf16_to_f32(W_down[(int64_t)j * d + c]);
        }
      } else {
        for (int32_t t = 0; t < nt; ++t) {
          int64_t cell = (int64_t)n * nt + t;
          for (int32_t s = 0; s < counts[cell]; ++s) {
            int32_t j = t * T + idx[cell * C + s];
            acc += bf16_to_f32(values[cell * C + s]) * bf16_to_f32(W_down[(int64_t)j * d + c]);
          }
        }
      }
      y[c] = acc;
    }
  }
}

EXPORT void oracle_round_bf16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(x[i]);
}

/* Backward of  L = sum(Y * dY) + lambda * sum|H|  with Y = H . W_down and
 * H = ReLU(X . W_in + b), fp32 dense loops over every (n, j), zero or not.
 *
 * dZ for selected rows: dH[n][j] = sum_c dY[n][c] * W_down[j][c] (c ascending);
 * dZ = dH + lambda where H[n][j] > 0, else 0.  H holds the selected rows. */
EXPORT void oracle_grad_hidden(const uint16_t* dY, const uint16_t* W_down, const uint16_t* H,
                               float lambda, const int32_t* rows, int32_t n_sel, int32_t d,
                               int32_t f, float* dH, float* dZ) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    const uint16_t* g = dY + (int64_t)rows[r] * d;
    for (int32_t j = 0; j < f; ++j) {
      const uint16_t* w = W_down + (int64_t)j * d;
      float acc = 0.0f;
      for (int32_t c = 0; c < d; ++c) acc += bf16_to_f32(g[c]) * bf16_to_f32(w[c]);
      float h = bf16_to_f32(H[(int64_t)r * f + j]);
      if (dH) dH[(int64_t)r * f + j] = acc;
      dZ[(int64_t)r * f + j] = (h > 0.0f) ? acc + lambda : 0.0f;
    }
  }
}

/* dX[r][k] = sum_j dZ[r][j] * W_inT[j][k] (j ascending). */
EXPORT void oracle_grad_input(const float* dZ, const uint16_t* W_inT, int32_t n_sel, int32_t d,
                              int32_t f, float* dX) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    for (int32_t k = 0; k < d; ++k) {
      float acc = 0.0f;
      for (int32_t j = 0; j < f; ++j) acc += dZ[(int64_t)r * f + j] * bf16_to_f32(W_inT[(int64_t)j * d + k]);
      dX[(int64_t)r * d + k] = acc;
    }
  }
}

/* Weight gradients for selected hidden units j, summing n ascending over all N
 * rows; H is the full [N][f] activation matrix:
 *   dW_down[j][c] = sum_n H[n][j] * dY[n][c]
 *   dW_inT[j][k]  = sum_n dZ[n][j] * X[n][k]
 *   db[j]         = sum_n dZ[n][j]
 * with dZ[n][j] recomputed from its definition. */
EXPORT void oracle_grad_weights(const uint16_t* X, const uint16_t* W_down, const uint16_t* H,
                                const uint16_t* dY, float lambda, int32_t N, int32_t d, int32_t f,
                                const int32_t* cols, int32_t n_cols, float* dW_inT,
                                float* dW_down, float* db) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t q = 0; q < n_cols; ++q) {
    int32_t j = cols[q];
    const uint16_t* w = W_down + (int64_t)j * d;
    float* gin = dW_inT + (int64_t)q * d;
    float* gdown = dW_down + (int64_t)q * d;
    float gb = 0.0f;
    for (int32_t k = 0; k < d; ++k) gin[k] = 0.0f;
    for (int32_t c = 0; c < d; ++c) gdown[c] = 0.0f;
    for (int32_t n = 0; n < N; ++n) {
      const uint16_t* g = dY + (int64_t)n * d;
      float h = bf16_to_f32(H[(int64_t)n * f + j]);
      float acc = 0.0f;
      for (int32_t c = 0; c < d; ++c) acc += bf16_to_f32(g[c]) * bf16_to_f32(w[c]);
      float dz = (h > 0.0f) ? acc + lambda : 0.0f;
      for (int32_t c = 0; c < d; ++c) gdown[c] += h * bf16_to_f32(g[c]);
      const uint16_t* x = X + (int64_t)n * d;
      for (int32_t k = 0; k < d; ++k) gin[k] += dz * bf16_to_f32(x[k]);
      gb += dz;
    }
    db[q] = gb;
  }
}

/* Backward of the gated layer  L = sum(Y * dY) + lambda * sum|H|  with
 * Y = H . W_down, H = bf16(g * u) where g = X . W_g + b > 0 (else +0) and
 * u = X . W_u (the Llama-style layer named "sparse_llama" on the
 * repo-explainer page, "The Repo's Two Jobs"; L1 on the activations from the
 * bayesiansapien note, TL;DR).  h's bf16 rounding is passed straight through
 * and the pattern is h != 0: where h != 0,
 *   dh = sum_c dY[n][c] * W_down[j][c] (c ascending) + lambda * sign(h),
 *   dG = dh * u,  dU = dh * g
 * (g and u recomputed as oracle_hidden_gated computes them); elsewhere dG and
 * dU are 0 -- including a (n, j) with g > 0 whose product rounds to zero. */
static void gated_point(const uint16_t* x, const uint16_t* wg, const uint16_t* wu, const uint16_t* bj,
                        const uint16_t* gy, const uint16_t* wd, uint16_t hbits, float lambda, int32_t d,
                        float* dg, float* du) {
  float h = bf16_to_f32(hbits);
  if (h == 0.0f) {
    *dg = 0.0f;
    *du = 0.0f;
    return;
  }
  float g = 0.0f, u = 0.0f, acc = 0.0f;
  for (int32_t k = 0; k < d; ++k) {
    g += bf16_to_f32(x[k]) * bf16_to_f32(wg[k]);
    u += bf16_to_f32(x[k]) * bf16_to_f32(wu[k]);
  }
  g += bf16_to_f32(*bj);
  for (int32_t c = 0; c < d; ++c) acc += bf16_to_f32(gy[c]) * bf16_to_f32(wd[c]);
  float dh = acc + (h > 0.0f ? lambda : -lambda);
  *dg = dh * u;
  *du = dh * g;
}

/* dG, dU for the selected rows ([n_sel][f] each); H holds the full [N][f]. */
EXPORT void oracle_grad_hidden_gated(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                     const uint16_t* b, const uint16_t* dY, const uint16_t* W_down,
                                     const uint16_t* H, float lambda, const int32_t* rows, int32_t n_sel,
                                     int32_t d, int32_t f, float* dG, float* dU) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    int32_t n = rows[r];
    for (int32_t j = 0; j < f; ++j)
      gated_point(X + (int64_t)n * d, W_gT + (int64_t)j * d, W_uT + (int64_t)j * d, b + j,
                  dY + (int64_t)n * d, W_down + (int64_t)j * d, H[(int64_t)n * f + j], lambda, d,
                  dG + (int64_t)r * f + j, dU + (int64_t)r * f + j);
  }
}

/* dX[r][k] = sum_j (dG[r][j] * W_gT[j][k] + dU[r][j] * W_uT[j][k]) (j ascending,
 * the gate's term then the up term). */
EXPORT void oracle_grad_input_gated(const float* dG, const float* dU, const uint16_t* W_gT,
                                    const uint16_t* W_uT, int32_t n_sel, int32_t d, int32_t f, float* dX) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_sel; ++r) {
    for (int32_t k = 0; k < d; ++k) {
      float acc = 0.0f;
      for (int32_t j = 0; j < f; ++j) {
        acc += dG[(int64_t)r * f + j] * bf16_to_f32(W_gT[(int64_t)j * d + k]);
        acc += dU[(int64_t)r * f + j] * bf16_to_f32(W_uT[(int64_t)j * d + k]);
      }
      dX[(int64_t)r * d + k] = acc;
    }
  }
}

/* Weight gradients of the gated layer for selected hidden units j, summing n
 * ascending over all N rows (dG, dU recomputed from their definition):
 *   dW_down[j][c] = sum_n H[n][j] * dY[n][c]
 *   dW_gT[j][k]   = sum_n dG[n][j] * X[n][k]
 *   dW_uT[j][k]   = sum_n dU[n][j] * X[n][k]
 *   db[j]         = sum_n dG[n][j]            (the bias sits on the gate) */
EXPORT void oracle_grad_weights_gated(const uint16_t* X, const uint16_t* W_gT, const uint16_t* W_uT,
                                      const uint16_t* b, const uint16_t* W_down, const uint16_t* H,
                                      const uint16_t* dY, float lambda, int32_t N, int32_t d, int32_t f,
                                      const int32_t* cols, int32_t n_cols, float* dW_gT, float* dW_uT,
                                      float* dW_down, float* db) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t q = 0; q < n_cols; ++q) {
    int32_t j = cols[q];
    float* gg = dW_gT + (int64_t)q * d;
    float* gu = dW_uT + (int64_t)q * d;
    float* gdown = dW_down + (int64_t)q * d;
    float gb = 0.0f;
    for (int32_t k = 0; k < d; ++k) gg[k] = gu[k] = gdown[k] = 0.0f;
    for (int32_t n = 0; n < N; ++n) {
      const uint16_t* x = X + (int64_t)n * d;
      const uint16_t* gy = dY + (int64_t)n * d;
      float h = bf16_to_f32(H[(int64_t)n * f + j]);
      float dg, du;
      gated_point(x, W_gT + (int64_t)j * d, W_uT + (int64_t)j * d, b + j, gy, W_down + (int64_t)j * d,
                  H[(int64_t)n * f + j], lambda, d, &dg, &du);
      for (int32_t c = 0; c < d; ++c) gdown[c] += h * bf16_to_f32(gy[c]);
      for (int32_t k = 0; k < d; ++k) {
        gg[k] += dg * bf16_to_f32(x[k]);
        gu[k] += du * bf16_to_f32(x[k]);
      }
      gb += dg;
    }
    db[q] = gb;
  }
}

/* Format invariants of a packed layer (no H needed).  Returns 0 when all hold,
 * else a code naming the first violated rule:
 *   1 count above C in a TwELL row      2 non-zero count in a fallback row
 *   3 index >= T                         4 indices not strictly increasing
 *   5 stored value equal to zero         6 padding slot not (+0.0, 0)
 *   7 row_fb / fb_rows not inverse (a row whose slot is past fb_cap, left
 *     unstored when the fallback overflowed, has no fb_rows entry)
 *   8 slots not numbered 0, 1, ... in ascending row order, or fb_rows not
 *     ascending
 *   9 number of fallback rows != n_fb */
EXPORT int32_t oracle_check_format(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                                   const int32_t* row_fb, const int32_t* fb_rows, int32_t n_fb,
                                   int32_t N, int32_t f, int32_t T, int32_t C, int32_t fb_cap) {
  const int32_t nt = f / T;
  int32_t seen_fb = 0;
  int misnumbered = 0;
  for (int32_t n = 0; n < N; ++n) {
    int is_fb = row_fb[n] >= 0;
    if (is_fb) {
      if (row_fb[n] != seen_fb) misnumbered = 1;
      seen_fb += 1;
      if (row_fb[n] < fb_cap && fb_rows[row_fb[n]] != n) return 7;
    } else if (row_fb[n] != -1) {
      return 7;
    }
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      int32_t cnt = counts[cell];
      if (is_fb && cnt != 0) return 2;
      if (cnt > C) return 1;
      for (int32_t s = 0; s < C; ++s) {
        uint16_t v = values[cell * C + s];
        uint8_t i = idx[cell * C + s];
        if (s < cnt) {
          if (i >= T) return 3;
          if (s > 0 && i <= idx[cell * C + s - 1]) return 4;
          if (bf16_to_f32(v) == 0.0f) return 5;
        } else if (v != 0 || i != 0) {
          return 6;
        }
      }
    }
  }
  if (misnumbered) return 8;
  for (int32_t s = 1; s < n_fb && s < fb_cap; ++s)
    if (fb_rows[s] <= fb_rows[s - 1]) return 8;
  if (seen_fb != n_fb) return 9;
  return 0;
}

/* Format invariants of the tile-granular hybrid.  Returns 0 when all hold,
 * else a code naming the first violated rule:
 *   1 count above C (and not 255)      3 index >= T
 *   4 indices not strictly increasing  5 stored value equal to zero
 *   6 padding slot not (+0.0, 0)       7 row_fb not -1
 *  10 dense tiles not numbered 0, 1, 2, ... in (row, tile) order
 *  11 number of dense tiles != min(n_dense, pool_cap)
 *  12 a dense tile with at most C non-zeros */
EXPORT int32_t oracle_check_format_tiles(const uint16_t* values, const uint8_t* idx, const uint8_t* counts,
                                         const int32_t* row_fb, const uint16_t* pool, int32_t n_dense, int32_t N,
                                         int32_t f, int32_t T, int32_t C, int32_t pool_cap) {
  const int32_t nt = f / T;
  int32_t next = 0;
  for (int32_t n = 0; n < N; ++n) {
    if (row_fb[n] != -1) return 7;
    for (int32_t t = 0; t < nt; ++t) {
      int64_t cell = (int64_t)n * nt + t;
      int32_t cnt = counts[cell];
      if (cnt == 255) {
        int32_t slot = (int32_t)values[cell * C] | ((int32_t)idx[cell * C] << 16);
        if (slot != next || slot >= pool_cap) return 10;
        int32_t nz = 0;
        for (int32_t i = 0; i < T; ++i)
          if (bf16_to_f32(pool[(int64_t)slot * T + i]) != 0.0f) nz += 1;
        if (nz <= C) return 12;
        for (int32_t s = 1; s < C; ++s)
          if (values[cell * C + s] != 0 || idx[cell * C + s] != 0) return 6;
        next += 1;
        continue;
      }
      if (cnt > C) return 1;
      for (int32_t s = 0; s < C; ++s) {
        uint16_t v = values[cell * C + s];
        uint8_t i = idx[cell * C + s];
        if (s < cnt) {
          if (i >= T) return 3;
          if (s > 0 && i <= idx[cell * C + s - 1]) return 4;
          if (bf16_to_f32(v) == 0.0f) return 5;
        } else if (v != 0 || i != 0) {
          return 6;
        }
      }
    }
  }
  if (next != (n_dense < pool_cap ? n_dense : pool_cap)) return 11;
  return 0;
}
