/*
 * Seeded synthetic inputs for the hierarchical KV cache resolver: top-k selection streams and host KV row
 * contents. This file holds no part of the resolution method (no hit test, no replacement, no copy policy);
 * it only draws the inputs that both the CPU oracle and the CUDA path consume.
 *
 * Random numbers:
 *   - splitmix64 (Vigna) expands a 64-bit seed into the 256-bit state of a xoshiro256** stream (Blackman and
 *     Vigna, "Scrambled linear pseudorandom number generators", 2018).
 *   - Bounded integers use the 128-bit multiply-high reduction (Lemire 2019) without the rejection step, so a
 *     draw is exactly one call of the stream.
 *   - Doubles in [0,1) take the top 53 bits of one draw.
 *
 * Selection stream of one (request, layer): step 0 draws k distinct tokens from the distribution. Each later
 * step keeps n_keep = floor((keep_pct*k + 50)/100) tokens of the previous selection, chosen uniformly without
 * replacement by a partial Fisher-Yates pass, then draws the other k - n_keep tokens from the distribution,
 * rejecting any token of the previous selection or one already drawn, and finally shuffles the row with a full
 * Fisher-Yates pass so that no consumer can assume sorted input. Churn steps use keep_pct = 0 (every token new).
 *
 * Distributions over positions 0..ctx-1: uniform, or Zipf(s) over recency ranks, where rank r (1..ctx) has
 * weight r^-s and rank 1 is the newest position ctx-1. Zipf draws invert the cumulative weight table by binary
 * search.
 *
 * Host rows: kind 0 fills bf16 values ~N(0,1) (Box-Muller, round-to-nearest-even from fp32), one counter-seeded
 * stream per row; kind 1 fills 64-bit words from a counter hash of (seed, layer, request, token, word), with
 * word 0 carrying (layer, request, token) so that every row is distinct.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static uint64_t sm64_next(uint64_t *x) {
  uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

typedef struct {
  uint64_t s[4];
} xo256;

static uint64_t rotl64(uint64_t x, int k) { return (x << k) | (x >> (64 - k)); }

static uint64_t xo_next(xo256 *r) {
  const uint64_t out = rotl64(r->s[1] * 5u, 7) * 9u;
  const uint64_t t = r->s[1] << 17;
  r->s[2] ^= r->s[0];
  r->s[3] ^= r->s[1];
  r->s[1] ^= r->s[2];
  r->s[0] ^= r->s[3];
  r->s[2] ^= t;
  r->s[3] = rotl64(r->s[3], 45);
  return out;
}

static void xo_seed(xo256 *r, uint64_t seed) {
  uint64_t x = seed;
  for (int i = 0; i < 4; ++i) r->s[i] = sm64_next(&x);
}

static uint64_t xo_below(xo256 *r, uint64_t n) {
  return (uint64_t)(((unsigned __int128)xo_next(r) * (unsigned __int128)n) >> 64);
}

static double xo_unit(xo256 *r) { return (double)(xo_next(r) >> 11) * (1.0 / 9007199254740992.0); }

/* Exported so that tests can pin the generator against the published reference outputs. */
uint64_t wl_splitmix64(uint64_t *state) { return sm64_next(state); }

void wl_xoshiro_sequence(uint64_t s0, uint64_t s1, uint64_t s2, uint64_t s3, int n, uint64_t *out) {
  xo256 r = {{s0, s1, s2, s3}};
  for (int i = 0; i < n; ++i) out[i] = xo_next(&r);
}

uint64_t wl_stream_seed(uint64_t seed, int32_t req, int32_t layer) {
  uint64_t x = seed ^ ((uint64_t)(uint32_t)req << 20) ^ (uint64_t)(uint32_t)layer;
  return sm64_next(&x);
}

enum { WL_UNIFORM = 0, WL_ZIPF = 1 };

typedef struct {
  int32_t ctx, dist;
  const double *cum; /* Zipf cumulative weights, cum[r-1] = sum_{i<=r} i^-s */
} wl_dist;

static int32_t draw_token(xo256 *r, const wl_dist *d) {
  if (d->dist == WL_UNIFORM) return (int32_t)xo_below(r, (uint64_t)d->ctx);
  const double u = xo_unit(r) * d->cum[d->ctx - 1];
  /* smallest rank index with cum > u */
  int32_t lo = 0, hi = d->ctx - 1;
  while (lo < hi) {
    int32_t mid = lo + (hi - lo) / 2;
    if (d->cum[mid] > u)
      hi = mid;
    else
      lo = mid + 1;
  }
  return d->ctx - 1 - lo; /* rank lo+1 -> position ctx-1-lo */
}

/*
 * Generate selections for layers [layer0, layer0+nlayers) x requests [req0, req0+nreq) over `steps` steps.
 * out: int32 [steps][nlayers][nreq][k]. churn: sorted list of step indices drawn with keep_pct = 0.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int wl_gen_selections(uint64_t seed, int32_t ctx, int32_t k, int32_t steps, int32_t keep_pct, int32_t dist,
                      double zipf_s, const int32_t *churn, int32_t n_churn, int32_t layer0, int32_t nlayers,
                      int32_t req0, int32_t nreq, int32_t *out) {
  if (ctx <= 0 || k <= 0 || 2 * (int64_t)k > ctx || steps <= 0 || keep_pct < 0 || keep_pct > 100) return -1;
  double *cum = NULL;
  if (dist == WL_ZIPF) {
    cum = (double *)malloc(sizeof(double) * (size_t)ctx);
    if (!cum) return -1;
    double acc = 0.0;
    for (int32_t r = 1; r <= ctx; ++r) {
      acc += pow((double)r, -zipf_s);
      cum[r - 1] = acc;
    }
  }
  wl_dist d = {ctx, dist, cum};
  uint8_t *mark = (uint8_t *)calloc((size_t)ctx, 1);
  int32_t *prev = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
  int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
  if (!mark || !prev || !tmp) {
    free(cum), free(mark), free(prev), free(tmp);
    return -1;
  }
  const size_t step_stride = (size_t)nlayers * (size_t)nreq * (size_t)k;
  for (int32_t li = 0; li < nlayers; ++li) {
    for (int32_t bi = 0; bi < nreq; ++bi) {
      xo256 r;
      xo_seed(&r, wl_stream_seed(seed, req0 + bi, layer0 + li));
      for (int32_t s = 0; s < steps; ++s) {
        int32_t *row = out + (size_t)s * step_stride + ((size_t)li * (size_t)nreq + (size_t)bi) * (size_t)k;
        int is_churn = 0;
        for (int32_t c = 0; c < n_churn; ++c) is_churn |= (churn[c] == s);
        const int32_t n_keep = (s == 0 || is_churn) ? 0 : (int32_t)(((int64_t)keep_pct * k + 50) / 100);
        if (s > 0) {
          memcpy(tmp, prev, sizeof(int32_t) * (size_t)k);
          for (int32_t i = 0; i < n_keep; ++i) {
            int32_t j = i + (int32_t)xo_below(&r, (uint64_t)(k - i));
            int32_t t = tmp[i];
            tmp[i] = tmp[j];
            tmp[j] = t;
            row[i] = tmp[i];
          }
          for (int32_t i = 0; i < k; ++i) mark[prev[i]] = 1;
        }
        for (int32_t i = 0; i < n_keep; ++i) mark[row[i]] = 1;
        for (int32_t i = n_keep; i < k; ++i) {
          int32_t t;
          do {
            t = draw_token(&r, &d);
          } while (mark[t]);
          mark[t] = 1;
          row[i] = t;
        }
        for (int32_t i = k - 1; i > 0; --i) {
          int32_t j = (int32_t)xo_below(&r, (uint64_t)(i + 1));
          int32_t t = row[i];
          row[i] = row[j];
          row[j] = t;
        }
        if (s > 0)
          for (int32_t i = 0; i < k; ++i) mark[prev[i]] = 0;
        for (int32_t i = 0; i < k; ++i) mark[row[i]] = 0;
        memcpy(prev, row, sizeof(int32_t) * (size_t)k);
      }
    }
  }
  free(cum), free(mark), free(prev), free(tmp);
  return 0;
}

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  const uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + bias) >> 16);
}

/*
 * Fill ntok consecutive host rows of (layer, req) starting at token tok0 into dst (ntok * row_bytes bytes).
 * kind 0: bf16 N(0,1); kind 1: hash words. row_bytes must be a multiple of 8 (kind 1) or 4 (kind 0).
 */
int wl_fill_rows(uint64_t seed, int32_t kind, int32_t row_bytes, int32_t layer, int32_t req, int64_t tok0,
                 int64_t ntok, uint8_t *dst) {
  if (row_bytes <= 0) return -1;
  if (kind == 0) {
    if (row_bytes % 4) return -1;
    const int32_t pairs = row_bytes / 4;
    for (int64_t t = 0; t < ntok; ++t) {
      const uint64_t tok = (uint64_t)(tok0 + t);
      xo256 r;
      xo_seed(&r, mix64(seed ^ 0xB5AD4ECEDA1CE2A9ull) ^ ((uint64_t)(uint32_t)layer << 48) ^
                      ((uint64_t)(uint32_t)req << 32) ^ tok);
      uint16_t *w = (uint16_t *)(dst + (size_t)t * (size_t)row_bytes);
      for (int32_t p = 0; p < pairs; ++p) {
        const double u1 = 1.0 - xo_unit(&r); /* (0,1] */
        const double u2 = xo_unit(&r);
        const double rad = sqrt(-2.0 * log(u1));
        const double ang = 6.283185307179586476925286766559 * u2;
        w[2 * p] = f32_to_bf16_rne((float)(rad * cos(ang)));
        w[2 * p + 1] = f32_to_bf16_rne((float)(rad * sin(ang)));
      }
    }
    return 0;
  }
  if (kind == 1) {
    if (row_bytes % 8) return -1;
    const int32_t words = row_bytes / 8;
    const uint64_t base = mix64(seed ^ 0x3C6EF372FE94F82Bull);
    for (int64_t t = 0; t < ntok; ++t) {
      const uint64_t tok = (uint64_t)(tok0 + t);
      uint64_t *w = (uint64_t *)(dst + (size_t)t * (size_t)row_bytes);
      const uint64_t rowkey = base ^ mix64(((uint64_t)(uint32_t)layer << 40) ^ ((uint64_t)(uint32_t)req << 24) ^
                                           (tok * 0x9E3779B97F4A7C15ull));
      w[0] = ((uint64_t)(uint16_t)layer << 48) | ((uint64_t)(uint16_t)req << 32) | (uint64_t)(uint32_t)tok;
      for (int32_t j = 1; j < words; ++j) w[j] = mix64(rowkey + (uint64_t)j * 0xD1B54A32D192ED03ull);
    }
    return 0;
  }
  return -1;
}
