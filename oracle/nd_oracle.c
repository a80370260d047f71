/*
 * nd_oracle.c -- plain fp64 CPU oracle for sliding-window + KV-sink attention
 * over a bounded int8 group-32 KV cache, and for the compressed-attention
 * variant (mean-pooled blocks rotated once at their midpoint).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load it (through oracle/__init__.py).  It shares
 * no header, helper, table or constant with the CUDA path.
 *
 * Every function writes out the plain definition it cites, with no blocking,
 * fusion or reordering: explicit dense masks, a dense softmax per query row,
 * fp64 arithmetic everywhere except the int8 codec, which is defined in fp32 so
 * that its integer codes are reproducible bit for bit (compile with
 * -ffp-contract=off and without fast-math).
 *
 * Sources (web pages, cited by title and section):
 *  [N1] "256-token滑动窗口+KV sink：Needle 2工具钉住机制源码分析", sections
 *       "256-token 滑动窗口：源码走读" (decode mask), "KV sink 如何「钉住」工具"
 *       (sink construction), "256 这个窗口宽度从哪来：内存预算计算器" (budget).
 *  [N2] "How the 256-Token Sliding Window Works with Tools as KV Sinks in
 *       Needle", sections "Effective KV Window: Bounding the Cache Size" and
 *       "KV Sinks for Tools: Pinning Critical Context".
 *  [C3] "Compressed attention and the copy probe", sections "Two kinds of
 *       columns, pooled blocks and exact recent keys" and "Pool before
 *       rotating, not after".
 *
 * Parity status: every exported function is pinned by a -m "not gpu" test
 * (closed forms, brute force, textbook reductions, the pages' printed values);
 * see tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int ndo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Masks                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * [N2] "KV Sinks for Tools" -- make_causal_packing_mask(seg_ids, prefix, window).
 * For every batch row b, query position q and key position k (positions are
 * the packed index 0..T-1):
 *   same block : seg[q] == seg[k] and seg[q] > 0   (segment 0 is padding)
 *   causal     : k <= q
 *   if window != 0 (a zero window switches the window term off):
 *     recent   : q - k < window
 *     sink     : prefix[k] > 0   (no prefix => no sinks)
 *     term     : recent or sink
 * mask[b][q][k] = 1 iff every term holds.  Output u8 [B][T][T]; the page's
 * head axis of size 1 is implicit (the mask is shared by every head).
 */
void ndo_causal_packing_mask(int B, int T, const int32_t *seg_ids,
                             const uint8_t *prefix, int window, uint8_t *mask) {
  for (int b = 0; b < B; ++b) {
    const int32_t *seg = seg_ids + (size_t)b * T;
    for (int q = 0; q < T; ++q) {
      for (int k = 0; k < T; ++k) {
        int same_block = (seg[q] == seg[k]) && (seg[q] > 0);
        int causal = (k <= q);
        int keep = same_block && causal;
        if (window != 0) {
          int recent = (q - k) < window;
          int sink = prefix ? (prefix[(size_t)b * T + k] > 0) : 0;
          keep = keep && (recent || sink);
        }
        mask[((size_t)b * T + q) * T + k] = (uint8_t)keep;
      }
    }
  }
}

/*
 * [N1] "256-token 滑动窗口：源码走读" -- the decode mask for one query position
 * against a list of cached key positions:
 *   recent = (qpos - kpos) < kv_window
 *   keep   = recent or sink[k]          (no sink array => recent alone)
 *   result = causal and keep,  causal = kpos <= qpos
 * The decode mask carries no segment term: one decode call serves one sequence.
 */
void ndo_decode_keep(int n_keys, int64_t qpos, const int64_t *kpos,
                     const uint8_t *sink, int kv_window, uint8_t *keep) {
  for (int k = 0; k < n_keys; ++k) {
    int recent = (qpos - kpos[k]) < (int64_t)kv_window;
    int pinned = sink ? (sink[k] != 0) : 0;
    int causal = kpos[k] <= qpos;
    keep[k] = (uint8_t)(causal && (recent || pinned));
  }
}

/*
 * [C3] "Two kinds of columns" calls attention_mask(length, window, 0) without
 * defining it.  Reading used here: the plain causal sliding window,
 * k <= q and q - k < window, with the third argument (sink count) zero.
 * Output u8 [length][length].
 */
void ndo_window_mask(int length, int window, uint8_t *mask) {
  for (int q = 0; q < length; ++q)
    for (int k = 0; k < length; ++k)
      mask[(size_t)q * length + k] = (uint8_t)((k <= q) && (q - k < window));
}

/*
 * [C3] "Two kinds of columns" -- compressed_mask(length, window, block).
 * Columns are [pooled blocks j = 0..length/block-1, exact tokens 0..length-1].
 *   pooled column j is visible from row q iff (j + 1) * block <= q - window + 1
 *   exact columns follow the windowed causal mask above.
 * Output u8 [length][length/block + length].
 */
void ndo_compressed_mask(int length, int window, int block, uint8_t *mask) {
  int nblk = length / block;
  int ncol = nblk + length;
  uint8_t *exact = (uint8_t *)malloc((size_t)length * length);
  ndo_window_mask(length, window, exact);
  for (int q = 0; q < length; ++q) {
    for (int j = 0; j < nblk; ++j)
      mask[(size_t)q * ncol + j] = (uint8_t)((j + 1) * block <= q - window + 1);
    for (int k = 0; k < length; ++k)
      mask[(size_t)q * ncol + nblk + k] = exact[(size_t)q * length + k];
  }
  free(exact);
}

/* ------------------------------------------------------------------------ */
/* Dense masked softmax attention                                             */
/* ------------------------------------------------------------------------ */

/*
 * Masked softmax attention, the definition the pages' mask is applied to
 * ([N2] "KV Sinks for Tools": a key is attended iff the mask holds; [N1]
 * "一张图看懂 Needle 2": GQA attention).
 *
 *   q    [B][Tq][Hq][d]      k, v [B][Tk][Hkv][d]      (fp64)
 *   mask [B][Tq][Tk] u8, batch stride mask_bstride elements (0 = shared)
 *   GQA: query head h reads KV head h / (Hq / Hkv) (contiguous groups).
 *   s_k  = (q . k_k) / sqrt(d)  for visible keys
 *   p_k  = exp(s_k - max_s) / sum_visible exp(s - max_s)
 *   out  = sum_k p_k v_k ;  lse = max_s + log(sum exp(s - max_s))
 * A row with no visible key gives out = 0 and lse = -inf.
 *
 * rows: NULL for every (b, t) row, else n_rows pairs (b, t); out is then
 * [n_rows][Hq][d] and lse [n_rows][Hq] (lse may be NULL).
 */
void ndo_attention(int B, int Tq, int Tk, int Hq, int Hkv, int d,
                   const double *q, const double *k, const double *v,
                   const uint8_t *mask, int64_t mask_bstride, int n_rows,
                   const int32_t *rows, double *out, double *lse) {
  int G = Hq / Hkv;
  int64_t total = rows ? (int64_t)n_rows : (int64_t)B * Tq;
  double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t item = 0; item < total * Hq; ++item) {
    int64_t r = item / Hq;
    int h = (int)(item % Hq);
    int b, t;
    if (rows) {
      b = rows[2 * r];
      t = rows[2 * r + 1];
    } else {
      b = (int)(r / Tq);
      t = (int)(r % Tq);
    }
    int hk = h / G;
    const double *qv = q + (((size_t)b * Tq + t) * Hq + h) * d;
    const uint8_t *mrow = mask + (size_t)b * mask_bstride + (size_t)t * Tk;
    double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    double smax = -INFINITY;
    for (int j = 0; j < Tk; ++j) {
      if (!mrow[j]) continue;
      const double *kv = k + (((size_t)b * Tk + j) * Hkv + hk) * d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c) dot += qv[c] * kv[c];
      s[j] = dot * scale;
      if (s[j] > smax) smax = s[j];
    }
    double *o = out + ((size_t)r * Hq + h) * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (smax == -INFINITY) {
      if (lse) lse[(size_t)r * Hq + h] = -INFINITY;
      free(s);
      continue;
    }
    double denom = 0.0;
    for (int j = 0; j < Tk; ++j)
      if (mrow[j]) denom += exp(s[j] - smax);
    for (int j = 0; j < Tk; ++j) {
      if (!mrow[j]) continue;
      double p = exp(s[j] - smax) / denom;
      const double *vv = v + (((size_t)b * Tk + j) * Hkv + hk) * d;
      for (int c = 0; c < d; ++c) o[c] += p * vv[c];
    }
    if (lse) lse[(size_t)r * Hq + h] = smax + log(denom);
    free(s);
  }
}

/* ------------------------------------------------------------------------ */
/* int8 group-32 KV codec                                                     */
/* ------------------------------------------------------------------------ */

/*
 * [N2] "Effective KV Window": each cached position stores 2*kv int8 bytes plus
 * 2*(kv/32)*4 bytes of scales, i.e. one fp32 scale per 32 contiguous channels
 * of K and of V.  The pages do not print the quantiser; the reading used
 * (symmetric absmax, fp32 arithmetic, so the codes are exact integers):
 *   amax  = max |x_c| over the 32 channels of a group
 *   scale = amax / 127                      (IEEE fp32 divide)
 *   code  = clamp(rint(x_c / scale), -127, 127)  (fp32 divide, ties to even)
 *   amax == 0: scale = 0 and every code is 0.
 * x [n][d] fp32 (d a multiple of 32) -> codes [n][d] int8, scales [n][d/32].
 */
void ndo_quant_g32(int n, int d, const float *x, int8_t *codes, float *scales) {
  int ng = d / 32;
  for (int i = 0; i < n; ++i) {
    for (int g = 0; g < ng; ++g) {
      const float *xg = x + (size_t)i * d + g * 32;
      float amax = 0.0f;
      for (int c = 0; c < 32; ++c) {
        float a = fabsf(xg[c]);
        if (a > amax) amax = a;
      }
      float scale = amax / 127.0f;
      scales[(size_t)i * ng + g] = scale;
      for (int c = 0; c < 32; ++c) {
        int8_t code = 0;
        if (amax != 0.0f) {
          float r = rintf(xg[c] / scale);
          if (r > 127.0f) r = 127.0f;
          if (r < -127.0f) r = -127.0f;
          code = (int8_t)r;
        }
        codes[(size_t)i * d + g * 32 + c] = code;
      }
    }
  }
}

/* The value a cached element stands for: code * scale, exact in fp64. */
double ndo_dequant(int8_t code, float scale) {
  return (double)code * (double)scale;
}

/* ------------------------------------------------------------------------ */
/* Bounded cache: pinned sink region + ring window                            */
/* ------------------------------------------------------------------------ */

/*
 * Cache layout (a data format shared by contract with the library, not code):
 *   codes  int8 [B][Hkv][sink_cap + ring_cap][d]
 *   scales fp32 [B][Hkv][sink_cap + ring_cap][d/32]
 *   slot s < sink_cap       : sink slot s (pinned, never evicted)
 *   slot sink_cap + r       : ring slot r, r < ring_cap
 *   per sequence b: sink_len, ring_start (ring slot of the oldest entry),
 *   ring_len (valid ring entries), seq_len (tokens seen = next position).
 *
 * [N1] "KV sink 如何「钉住」工具" / [N2] "KV Sinks for Tools": pinned positions
 * are never evicted; the rest of the cache keeps the most recent window.
 * Reading for the ring (the pages give none): a new ring token goes to ring
 * slot (ring_start + ring_len) mod ring_cap; when the ring is full it
 * overwrites the oldest entry and ring_start advances.  A sink token goes to
 * sink slot sink_len and is accepted only while the ring is empty and
 * sink_len < sink_cap (the sink is a prefix).  Every append takes position
 * seq_len.  Returns the number of rejected sink appends.
 *
 * k_new, v_new: fp32 [B][Hkv][d] (the bf16 token widened exactly).
 */
int ndo_kv_append(int B, int Hkv, int d, int sink_cap, int ring_cap,
                  int8_t *k_codes, float *k_scale, int8_t *v_codes,
                  float *v_scale, int32_t *sink_len, int32_t *ring_start,
                  int32_t *ring_len, int32_t *seq_len, const float *k_new,
                  const float *v_new, int to_sink) {
  int ng = d / 32;
  int nslot = sink_cap + ring_cap;
  int rejected = 0;
  for (int b = 0; b < B; ++b) {
    int slot;
    if (to_sink) {
      if (ring_len[b] != 0 || sink_len[b] >= sink_cap) {
        ++rejected;
        continue;
      }
      slot = sink_len[b];
      sink_len[b] += 1;
    } else {
      if (ring_len[b] < ring_cap) {
        slot = sink_cap + (ring_start[b] + ring_len[b]) % ring_cap;
        ring_len[b] += 1;
      } else {
        slot = sink_cap + ring_start[b];
        ring_start[b] = (ring_start[b] + 1) % ring_cap;
      }
    }
    seq_len[b] += 1;
    for (int h = 0; h < Hkv; ++h) {
      size_t row = ((size_t)b * Hkv + h) * nslot + slot;
      ndo_quant_g32(1, d, k_new + ((size_t)b * Hkv + h) * d, k_codes + row * d,
                    k_scale + row * ng);
      ndo_quant_g32(1, d, v_new + ((size_t)b * Hkv + h) * d, v_codes + row * d,
                    v_scale + row * ng);
    }
  }
  return rejected;
}

/*
 * Absolute position held by every slot of sequence b, or -1 for an empty slot,
 * under the append rule above: sink slot s holds position s; the ring's
 * entries, oldest first, hold the ring_len positions that end at seq_len - 1.
 */
void ndo_slot_positions(int sink_cap, int ring_cap, int32_t sink_len,
                        int32_t ring_start, int32_t ring_len, int32_t seq_len,
                        int64_t *kpos, uint8_t *is_sink) {
  for (int s = 0; s < sink_cap + ring_cap; ++s) {
    kpos[s] = -1;
    is_sink[s] = 0;
  }
  for (int s = 0; s < sink_len; ++s) {
    kpos[s] = s;
    is_sink[s] = 1;
  }
  for (int i = 0; i < ring_len; ++i) {
    int r = (ring_start + i) % ring_cap;
    kpos[sink_cap + r] = (int64_t)seq_len - ring_len + i;
  }
}

/*
 * One decode step ([N1] "256-token 滑动窗口：源码走读"): the query of sequence
 * b sits at position seq_len[b] - 1 (the newest cached token, appended before
 * attending).  Every occupied slot is a key; its mask is ndo_decode_keep with
 * the sink flag of its region; K and V are the dequantised codes.  The
 * attention itself is ndo_attention with one query row.
 *   q [B][Hq][d] fp64 -> out [B][Hq][d] fp64, lse [B][Hq] (may be NULL).
 */
void ndo_decode(int B, int Hq, int Hkv, int d, int sink_cap, int ring_cap,
                const double *q, const int8_t *k_codes, const float *k_scale,
                const int8_t *v_codes, const float *v_scale,
                const int32_t *sink_len, const int32_t *ring_start,
                const int32_t *ring_len, const int32_t *seq_len, int window,
                double *out, double *lse) {
  int ng = d / 32;
  int nslot = sink_cap + ring_cap;
  /* Sequences are independent: with more than one, each thread takes whole
   * sequences (the attention inside then runs on that thread alone); every
   * sequence's arithmetic is the same either way. */
#pragma omp parallel for schedule(dynamic, 1) if (B > 1)
  for (int b = 0; b < B; ++b) {
    int64_t *kpos = (int64_t *)malloc(sizeof(int64_t) * nslot);
    uint8_t *is_sink = (uint8_t *)malloc(nslot);
    uint8_t *keep = (uint8_t *)malloc(nslot);
    double *kd = (double *)malloc(sizeof(double) * (size_t)nslot * Hkv * d);
    double *vd = (double *)malloc(sizeof(double) * (size_t)nslot * Hkv * d);
    ndo_slot_positions(sink_cap, ring_cap, sink_len[b], ring_start[b],
                       ring_len[b], seq_len[b], kpos, is_sink);
    int64_t qpos = (int64_t)seq_len[b] - 1;
    ndo_decode_keep(nslot, qpos, kpos, is_sink, window, keep);
    for (int s = 0; s < nslot; ++s)
      if (kpos[s] < 0) keep[s] = 0; /* empty slot: no key there */
    /* Gather keys in [slot][Hkv][d] order, the layout ndo_attention reads. */
    for (int s = 0; s < nslot; ++s)
      for (int h = 0; h < Hkv; ++h) {
        size_t row = ((size_t)b * Hkv + h) * nslot + s;
        for (int c = 0; c < d; ++c) {
          kd[((size_t)s * Hkv + h) * d + c] =
              ndo_dequant(k_codes[row * d + c], k_scale[row * ng + c / 32]);
          vd[((size_t)s * Hkv + h) * d + c] =
              ndo_dequant(v_codes[row * d + c], v_scale[row * ng + c / 32]);
        }
      }
    ndo_attention(1, 1, nslot, Hq, Hkv, d, q + (size_t)b * Hq * d, kd, vd, keep,
                  0, 0, NULL, out + (size_t)b * Hq * d,
                  lse ? lse + (size_t)b * Hq : NULL);
    free(kpos);
    free(is_sink);
    free(keep);
    free(kd);
    free(vd);
  }
}

/* ------------------------------------------------------------------------ */
/* Compressed attention: pooling and rotary embedding                         */
/* ------------------------------------------------------------------------ */

/*
 * [C3] "Compressed attention and the copy probe": every block of `block`
 * consecutive keys becomes one averaged key, same for values.  Reading of the
 * unprinted pool_blocks: the arithmetic mean of positions jb .. jb+b-1, for
 * j < T / block (a trailing partial block is dropped, as length // block in
 * compressed_mask implies).
 *   x [B][T][H][d] -> out [B][T/block][H][d]
 */
void ndo_pool_blocks(int B, int T, int H, int d, int block, const double *x,
                     double *out) {
  int nblk = T / block;
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < nblk; ++j)
      for (int h = 0; h < H; ++h)
        for (int c = 0; c < d; ++c) {
          double sum = 0.0;
          for (int i = 0; i < block; ++i)
            sum += x[(((size_t)b * T + (size_t)j * block + i) * H + h) * d + c];
          out[(((size_t)b * nblk + j) * H + h) * d + c] = sum / block;
        }
}

/*
 * Rotary embedding, rotate-half convention (the pages call apply_rope without
 * printing it): for channel pair (i, i + d/2), i < d/2, at position m,
 *   angle   = m * theta^(-2i/d)
 *   x'_i       = x_i cos(angle) - x_{i+d/2} sin(angle)
 *   x'_{i+d/2} = x_{i+d/2} cos(angle) + x_i sin(angle)
 * x [B][T][H][d], pos [T] (one position per sequence index) -> out (same).
 */
void ndo_rope(int B, int T, int H, int d, const double *x, const int64_t *pos,
              double theta, double *out) {
  int half = d / 2;
  for (int b = 0; b < B; ++b)
    for (int t = 0; t < T; ++t)
      for (int h = 0; h < H; ++h) {
        const double *xi = x + (((size_t)b * T + t) * H + h) * d;
        double *xo = out + (((size_t)b * T + t) * H + h) * d;
        for (int i = 0; i < half; ++i) {
          double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
          double angle = (double)pos[t] * inv_freq;
          double c = cos(angle), s = sin(angle);
          double x1 = xi[i], x2 = xi[i + half];
          xo[i] = x1 * c - x2 * s;
          xo[i + half] = x2 * c + x1 * s;
        }
      }
}

/*
 * [C3] "Pool before rotating, not after" (_compress): pool K and V before any
 * rotation, rotate each pooled key once at its block midpoint
 *   m_j = min(j * block + block / 2, table_len - 1)   (integer block / 2)
 * rotate q and k at their own positions 0..T-1, then concatenate along the
 * sequence axis: K' = [pooled K ; K], V' = [pooled V ; V].
 * theta == 0 means no rotary table: nothing is rotated.
 *   q, k, v [B][T][H][d]
 *   q_out [B][T][H][d]; k_out, v_out [B][T/block + T][H][d]
 */
void ndo_compress(int B, int T, int H, int d, int block, double theta,
                  int table_len, const double *q, const double *k,
                  const double *v, double *q_out, double *k_out,
                  double *v_out) {
  int nblk = T / block;
  int ncol = nblk + T;
  size_t plane = (size_t)H * d;
  double *pk = (double *)malloc(sizeof(double) * (size_t)B * (nblk > 0 ? nblk : 1) * plane);
  double *pv = (double *)malloc(sizeof(double) * (size_t)B * (nblk > 0 ? nblk : 1) * plane);
  double *kr = (double *)malloc(sizeof(double) * (size_t)B * T * plane);
  ndo_pool_blocks(B, T, H, d, block, k, pk);
  ndo_pool_blocks(B, T, H, d, block, v, pv);
  if (theta != 0.0) {
    int64_t *mid = (int64_t *)malloc(sizeof(int64_t) * (nblk > 0 ? nblk : 1));
    int64_t *own = (int64_t *)malloc(sizeof(int64_t) * (T > 0 ? T : 1));
    for (int j = 0; j < nblk; ++j) {
      int64_t m = (int64_t)j * block + block / 2;
      mid[j] = m < table_len - 1 ? m : table_len - 1;
    }
    for (int t = 0; t < T; ++t) own[t] = t;
    double *pkr = (double *)malloc(sizeof(double) * (size_t)B * (nblk > 0 ? nblk : 1) * plane);
    ndo_rope(B, nblk, H, d, pk, mid, theta, pkr);
    memcpy(pk, pkr, sizeof(double) * (size_t)B * nblk * plane);
    free(pkr);
    ndo_rope(B, T, H, d, q, own, theta, q_out);
    ndo_rope(B, T, H, d, k, own, theta, kr);
    free(mid);
    free(own);
  } else {
    memcpy(q_out, q, sizeof(double) * (size_t)B * T * plane);
    memcpy(kr, k, sizeof(double) * (size_t)B * T * plane);
  }
  for (int b = 0; b < B; ++b) {
    for (int j = 0; j < nblk; ++j) {
      memcpy(k_out + ((size_t)b * ncol + j) * plane, pk + ((size_t)b * nblk + j) * plane, sizeof(double) * plane);
      memcpy(v_out + ((size_t)b * ncol + j) * plane, pv + ((size_t)b * nblk + j) * plane, sizeof(double) * plane);
    }
    for (int t = 0; t < T; ++t) {
      memcpy(k_out + ((size_t)b * ncol + nblk + t) * plane, kr + ((size_t)b * T + t) * plane, sizeof(double) * plane);
      memcpy(v_out + ((size_t)b * ncol + nblk + t) * plane, v + ((size_t)b * T + t) * plane, sizeof(double) * plane);
    }
  }
  free(pk);
  free(pv);
  free(kr);
}

/* ------------------------------------------------------------------------ */
/* KV budget window                                                           */
/* ------------------------------------------------------------------------ */

/*
 * [N1] "256 这个窗口宽度从哪来" and [N2] "Effective KV Window": constants
 *   budget bytes = 11 MiB + 512 KiB, group = 32, minimum window = 160
 * and kv_budget_window:
 *   head_dim = (attn_dim or d_model) / num_heads      (attn_dim 0 = unset)
 *   kv       = num_kv_heads * head_dim
 *   per_pos  = L * (2 kv + 2 (kv / 32) * 4) + sites * (d_model + 32 * 4)
 *   window   = ((budget / per_pos) / 32) * 32
 *   result   = max(160, min(window, max_seq_len))
 * All divisions are floor divisions of non-negative integers.
 * Returns -1 when the configuration divides by zero.
 */
int64_t ndo_kv_budget_window(int64_t d_model, int64_t attn_dim,
                             int64_t num_heads, int64_t num_kv_heads,
                             int64_t num_layers, int64_t sites,
                             int64_t max_seq_len) {
  const int64_t budget_bytes = 11LL * 1024 * 1024 + 512LL * 1024;
  const int64_t group = 32;
  const int64_t window_min = 160;
  if (num_heads <= 0) return -1;
  int64_t head_dim = (attn_dim ? attn_dim : d_model) / num_heads;
  int64_t kv = num_kv_heads * head_dim;
  int64_t per_pos = num_layers * (2 * kv + 2 * (kv / group) * 4) +
                    sites * (d_model + group * 4);
  if (per_pos <= 0) return -1;
  int64_t window = (budget_bytes / per_pos) / group * group;
  int64_t capped = window < max_seq_len ? window : max_seq_len;
  return capped > window_min ? capped : window_min;
}

/*
 * [N2] "Effective KV Window": effective_kv_window = min(budget, kv_window)
 * when kv_window is set (non-zero), else the budget window.
 */
int64_t ndo_effective_kv_window(int64_t budget_window, int64_t kv_window) {
  if (kv_window) return budget_window < kv_window ? budget_window : kv_window;
  return budget_window;
}
