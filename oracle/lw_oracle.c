/*
 * lw_oracle.c -- plain CPU reference for entropy-coded weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no code, header, table or
 * constant with the CUDA library: it is written from the method's definition,
 * slowly and plainly, so that a reader can check it by eye.
 *
 * What it follows:
 *  - "LazyWeights: Decode-on-Demand Edge LLMs", section "2 . Code them" and
 *    Fig. 3(a): one length-limited (11-bit) Huffman table per matrix; a 64x256
 *    tile is 32 lanes of two rows; each lane is one stream of 32-bit words and
 *    the lanes' words are interleaved; per-tile offsets let a tile start alone.
 *  - same page, section "3 . Decode on demand" and Fig. 3(b): a lane compares
 *    an 11-bit peek against per-length limits, adds the length's offset to
 *    index the symbol table and shifts by the code length.
 *  - Length limiting: package-merge (Larmore & Hirschberg, 1990), the
 *    optimal length-limited prefix code.  The pages only say "length-limited".
 *  - Canonical code assignment: the rule of RFC 1951 section 3.2.2 (shorter
 *    codes first, ties by ascending symbol value).
 *
 * Conventions (the bundle format, which the library implements separately):
 *  - codes are written MSB-first: stream bit p lives in word p/32 at bit
 *    31 - p%32;
 *  - every lane of a tile is zero-padded to the tile's longest lane, W_t words;
 *  - word j of lane l of tile t sits at words[(tile_off[t] + j) * 32 + l];
 *  - tile_off has n_tiles + 1 entries, counted in rows of 32 words.
 *
 * All functions return 0 on success and a negative value on bad input.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_MAXLEN 11        /* the pages' code-length limit */
#define OR_MAXALPHA 256     /* pair symbols of two 4-bit codes */

/* ------------------------------------------------------------------------ */
/* Package-merge (coin collector) for optimal lengths <= lmax.               */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint64_t weight;
  int leaf;      /* 1: a single coin of symbol `sym`; 0: a package of two */
  int sym;       /* leaf only */
  int child_a;   /* package only: indices into the next-deeper list */
  int child_b;
} pm_item;

static const uint64_t *g_sort_counts;

static int cmp_leaf(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb;
  if (g_sort_counts[a] != g_sort_counts[b])
    return g_sort_counts[a] < g_sort_counts[b] ? -1 : 1;
  return a - b; /* ties by symbol value */
}

static void pm_count(pm_item **lists, int depth, int idx, int lmax,
                     uint8_t *len) {
  const pm_item *it = &lists[depth][idx];
  if (it->leaf) {
    len[it->sym]++;
    return;
  }
  /* a package at depth d was made from two items of depth d+1 */
  pm_count(lists, depth + 1, it->child_a, lmax, len);
  pm_count(lists, depth + 1, it->child_b, lmax, len);
}

/*
 * Optimal code lengths with every length <= lmax.
 * counts[alpha]: symbol frequencies.  len[alpha] receives the lengths; a
 * symbol that never occurs gets length 0.  A lone symbol gets length 1.
 */
int or_code_lengths(const uint64_t *counts, int alpha, int lmax,
                    uint8_t *len) {
  if (alpha <= 0 || alpha > 65536 || lmax < 1 || lmax > 30) return -1;
  memset(len, 0, (size_t)alpha);
  int n = 0, only = -1;
  for (int s = 0; s < alpha; s++)
    if (counts[s]) { n++; only = s; }
  if (n == 0) return 0;
  if (n == 1) { len[only] = 1; return 0; }
  if (lmax < 31 && ((uint64_t)1 << lmax) < (uint64_t)n) return -2;

  int *leaves = (int *)malloc(sizeof(int) * (size_t)n);
  for (int s = 0, k = 0; s < alpha; s++)
    if (counts[s]) leaves[k++] = s;
  g_sort_counts = counts;
  qsort(leaves, (size_t)n, sizeof(int), cmp_leaf);

  /* lists[d], d = lmax (coins of value 2^-lmax) up to d = 1 (2^-1). */
  pm_item **lists = (pm_item **)calloc((size_t)lmax + 2, sizeof(pm_item *));
  int *sizes = (int *)calloc((size_t)lmax + 2, sizeof(int));
  lists[lmax] = (pm_item *)malloc(sizeof(pm_item) * (size_t)n);
  for (int i = 0; i < n; i++) {
    pm_item it = {counts[leaves[i]], 1, leaves[i], -1, -1};
    lists[lmax][i] = it;
  }
  sizes[lmax] = n;
  for (int d = lmax - 1; d >= 1; d--) {
    int npk = sizes[d + 1] / 2;
    lists[d] = (pm_item *)malloc(sizeof(pm_item) * (size_t)(n + npk));
    int i = 0, j = 0, k = 0;
    /* merge the sorted leaves with the packages of the deeper list; on equal
       weight the leaf goes first */
    while (i < n || j < npk) {
      uint64_t pw = 0;
      if (j < npk)
        pw = lists[d + 1][2 * j].weight + lists[d + 1][2 * j + 1].weight;
      if (j >= npk || (i < n && counts[leaves[i]] <= pw)) {
        pm_item it = {counts[leaves[i]], 1, leaves[i], -1, -1};
        lists[d][k++] = it;
        i++;
      } else {
        pm_item it = {pw, 0, -1, 2 * j, 2 * j + 1};
        lists[d][k++] = it;
        j++;
      }
    }
    sizes[d] = k;
  }
  /* the cheapest 2n-2 items at value 1/2 add up to n-1 */
  for (int i = 0; i < 2 * n - 2; i++) pm_count(lists, 1, i, lmax, len);

  for (int d = 1; d <= lmax; d++) free(lists[d]);
  free(lists);
  free(sizes);
  free(leaves);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Canonical codes (RFC 1951 section 3.2.2).                                 */
/* ------------------------------------------------------------------------ */

int or_canonical_codes(const uint8_t *len, int alpha, uint32_t *code) {
  uint32_t bl_count[32] = {0}, next_code[32] = {0};
  int maxlen = 0;
  for (int s = 0; s < alpha; s++) {
    if (len[s] > 30) return -1;
    if (len[s]) bl_count[len[s]]++;
    if (len[s] > maxlen) maxlen = len[s];
  }
  uint32_t c = 0;
  bl_count[0] = 0;
  for (int b = 1; b <= maxlen; b++) {
    c = (c + bl_count[b - 1]) << 1;
    next_code[b] = c;
  }
  for (int s = 0; s < alpha; s++) {
    code[s] = 0;
    if (len[s]) code[s] = next_code[len[s]]++;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Decoder tables for the comparator rule.                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint32_t first_code[OR_MAXLEN + 2]; /* first canonical code of length L */
  uint32_t count[OR_MAXLEN + 2];      /* number of codes of length L */
  uint32_t limit[OR_MAXLEN + 2];      /* (first_code+count) << (11-L) */
  uint32_t base[OR_MAXLEN + 2];       /* symbols with length < L */
  uint16_t sorted[OR_MAXALPHA];
  int nsym;
} or_tables;

static int build_tables(const uint8_t *len, int alpha, or_tables *t) {
  memset(t, 0, sizeof(*t));
  if (alpha > OR_MAXALPHA) return -1;
  for (int s = 0; s < alpha; s++) {
    if (len[s] > OR_MAXLEN) return -1;
    if (len[s]) t->count[len[s]]++;
  }
  uint32_t c = 0;
  for (int L = 1; L <= OR_MAXLEN; L++) {
    c = (c + (L > 1 ? t->count[L - 1] : 0)) << (L > 1 ? 1 : 0);
    t->first_code[L] = c;
  }
  uint32_t b = 0;
  for (int L = 1; L <= OR_MAXLEN; L++) {
    t->base[L] = b;
    b += t->count[L];
    t->limit[L] = (t->first_code[L] + t->count[L]) << (OR_MAXLEN - L);
  }
  /* symbols in canonical order: by length, then by symbol value */
  int k = 0;
  for (int L = 1; L <= OR_MAXLEN; L++)
    for (int s = 0; s < alpha; s++)
      if (len[s] == L) t->sorted[k++] = (uint16_t)s;
  t->nsym = k;
  return 0;
}

/* Exported for the tests: limits, first codes, counts and bases, L = 0..11. */
int or_decoder_tables(const uint8_t *len, int alpha, uint32_t *first_code,
                      uint32_t *count, uint32_t *limit, uint32_t *base,
                      uint16_t *sorted) {
  or_tables *t = (or_tables *)malloc(sizeof(or_tables));
  int rc = build_tables(len, alpha, t);
  if (rc == 0) {
    for (int L = 0; L <= OR_MAXLEN; L++) {
      first_code[L] = t->first_code[L];
      count[L] = t->count[L];
      limit[L] = t->limit[L];
      base[L] = t->base[L];
    }
    memcpy(sorted, t->sorted, sizeof(uint16_t) * (size_t)t->nsym);
  }
  free(t);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Lane streams: encode (pack + interleave) and decode.                       */
/* ------------------------------------------------------------------------ */

static void put_bits(uint32_t *lane_words, uint64_t *bitpos, uint32_t code,
                     int L) {
  for (int i = L - 1; i >= 0; i--) {          /* MSB of the code first */
    uint32_t bit = (code >> i) & 1u;
    uint64_t p = *bitpos;
    if (bit) lane_words[p / 32] |= 1u << (31 - (p % 32));
    (*bitpos)++;
  }
}

/*
 * Pack lanes.  syms[(t*32 + l) * maxsym + i] is symbol i of lane l of tile t;
 * nsym[t*32 + l] symbols are used.  Pass words == NULL to size only: the
 * function always fills tile_off[n_tiles+1] and lane_bits[n_tiles*32].
 * words must hold tile_off[n_tiles] * 32 entries.
 */
int or_pack_lanes(const uint8_t *len, int alpha, const uint16_t *syms,
                  const int32_t *nsym, int64_t n_tiles, int maxsym,
                  uint32_t *tile_off, uint16_t *lane_bits, uint32_t *words) {
  uint32_t *code = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)alpha);
  if (or_canonical_codes(len, alpha, code)) { free(code); return -1; }
  /* a lane holds at most maxsym codes of at most 11 bits */
  int lane_cap = (maxsym * OR_MAXLEN + 31) / 32 + 1;
  uint32_t *lane = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)lane_cap);
  tile_off[0] = 0;
  for (int64_t t = 0; t < n_tiles; t++) {
    uint32_t wt = 0;
    for (int l = 0; l < 32; l++) {
      uint64_t bits = 0;
      const uint16_t *s = syms + (t * 32 + l) * maxsym;
      for (int i = 0; i < nsym[t * 32 + l]; i++) {
        if (s[i] >= alpha || len[s[i]] == 0) { free(code); free(lane); return -2; }
        bits += len[s[i]];
      }
      lane_bits[t * 32 + l] = (uint16_t)bits;
      uint32_t w = (uint32_t)((bits + 31) / 32);
      if (w > wt) wt = w;
    }
    tile_off[t + 1] = tile_off[t] + wt;
    if (!words) continue;
    for (int l = 0; l < 32; l++) {
      memset(lane, 0, sizeof(uint32_t) * (size_t)lane_cap);
      uint64_t p = 0;
      const uint16_t *s = syms + (t * 32 + l) * maxsym;
      for (int i = 0; i < nsym[t * 32 + l]; i++)
        put_bits(lane, &p, code[s[i]], len[s[i]]);
      for (uint32_t j = 0; j < wt; j++)
        words[((uint64_t)tile_off[t] + j) * 32 + l] = lane[j];
    }
  }
  free(code);
  free(lane);
  return 0;
}

/* bit p of lane l of a tile whose rows start at `rows`, W_t rows long;
   bits past the tile read as zero */
static uint32_t get_bit(const uint32_t *rows, uint32_t wt, int l, uint64_t p) {
  uint64_t j = p / 32;
  if (j >= wt) return 0;
  return (rows[j * 32 + l] >> (31 - (p % 32))) & 1u;
}

/*
 * Decode every lane with the comparator rule.  out[(t*32+l)*maxsym + i]
 * receives symbol i; bits_used[t*32+l] the number of bits consumed.
 * Returns -3 if a peek matches no code (corrupt stream).
 */
int or_decode_lanes(const uint8_t *len, int alpha, const uint32_t *words,
                    const uint32_t *tile_off, int64_t n_tiles,
                    const int32_t *nsym, int maxsym, uint16_t *out,
                    uint32_t *bits_used) {
  or_tables *tb = (or_tables *)malloc(sizeof(or_tables));
  if (build_tables(len, alpha, tb)) { free(tb); return -1; }
  int rc = 0;
  for (int64_t t = 0; t < n_tiles && rc == 0; t++) {
    const uint32_t *rows = words + (uint64_t)tile_off[t] * 32;
    uint32_t wt = tile_off[t + 1] - tile_off[t];
    for (int l = 0; l < 32 && rc == 0; l++) {
      uint64_t p = 0;
      for (int i = 0; i < nsym[t * 32 + l]; i++) {
        /* the next 11 bits of the lane, first bit most significant */
        uint32_t peek = 0;
        for (int k = 0; k < OR_MAXLEN; k++)
          peek = (peek << 1) | get_bit(rows, wt, l, p + (uint64_t)k);
        /* smallest length whose limit lies above the peek */
        int L = 0;
        for (int c = 1; c <= OR_MAXLEN; c++)
          if (peek < tb->limit[c]) { L = c; break; }
        if (L == 0) { rc = -3; break; }
        uint32_t code = peek >> (OR_MAXLEN - L);
        uint32_t idx = tb->base[L] + (code - tb->first_code[L]);
        if (idx >= (uint32_t)tb->nsym) { rc = -3; break; }
        out[(t * 32 + l) * maxsym + i] = tb->sorted[idx];
        p += (uint64_t)L;
      }
      bits_used[t * 32 + l] = (uint32_t)p;
    }
  }
  free(tb);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Dot products in double precision.                                          */
/* ------------------------------------------------------------------------ */

/* y[b*n + r] = sum_k w[r*k_dim + k] * x[b*k_dim + k], k ascending, in fp64 */
void or_gemm_f64(const double *w, const double *x, int64_t n, int64_t k_dim,
                 int batch, double *y) {
  for (int b = 0; b < batch; b++)
    for (int64_t r = 0; r < n; r++) {
      double acc = 0.0;
      for (int64_t k = 0; k < k_dim; k++)
        acc += w[r * k_dim + k] * x[(int64_t)b * k_dim + k];
      y[(int64_t)b * n + r] = acc;
    }
}
