/*
 * A plain C11 caller of liblw's host entry points: no Python, no PyTorch,
 * only include/lw.h and the shared library.  Compiled and run on the CPU by
 * tests/test_c_consumer.py.
 *
 * It builds a 4-bit bundle of a 128 x 512 matrix of codes drawn from a
 * fixed linear congruential generator, checks its sections against the
 * header's contract (one 128-byte word row per tile step, tile offsets
 * starting at 0 and ending at the word count, code lengths within 11 bits,
 * a complete prefix code: the Kraft sum of the table's code lengths is
 * exactly 1), validates them, round-trips the bundle through its byte-string
 * form, and checks that a corrupted string is refused.  Prints "ok" and
 * exits 0, or names the failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "lw.h"

#define N 128
#define K 512

static int failed(const char* what) {
  printf("FAILED: %s (%s)\n", what, lw_last_error());
  return 1;
}

static uint32_t lcg(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;
  return *s >> 8;
}

int main(void) {
  static uint8_t codes[N * K];
  static uint16_t scales[N * (K / 256)], mins[N * (K / 256)];
  uint32_t seed = 12345u;
  for (int i = 0; i < N * K; ++i) {
    /* a peaked distribution over 0..15: the sum of three small draws */
    codes[i] = (uint8_t)((lcg(&seed) % 6) + (lcg(&seed) % 6) + (lcg(&seed) % 6));
  }
  for (int i = 0; i < N * (K / 256); ++i) {
    scales[i] = 0x2000u + (uint16_t)(lcg(&seed) % 0x400); /* fp16 in [2^-7, 2^-6) */
    mins[i] = 0xA000u + (uint16_t)(lcg(&seed) % 0x400);   /* small negative fp16 */
  }

  lw_desc d = {LW_FMT_Q4_PAIR, 0, N, K};
  lw_bundle* b = NULL;
  if (lw_encode_bundle(&d, codes, scales, mins, &b) != LW_OK || !b) return failed("encode");

  lw_sections s;
  if (lw_bundle_sections(b, &s) != LW_OK) return failed("sections");
  const uint64_t n_tiles = (N / 64) * (K / 256);
  if (s.n_tiles != n_tiles) return failed("tile count");
  if (s.bytes[LW_SEC_TILE_OFF] != (n_tiles + 1) * 4) return failed("tile_off size");
  const uint32_t* off = (const uint32_t*)s.ptr[LW_SEC_TILE_OFF];
  if (off[0] != 0 || (uint64_t)off[n_tiles] * 128 != s.bytes[LW_SEC_WORDS])
    return failed("tile offsets against the word count");
  if (s.max_len < 1 || s.max_len > LW_MAX_CODE_LEN || s.min_len > s.max_len)
    return failed("code length span");
  if (s.bytes[LW_SEC_TABLE] != sizeof(lw_table)) return failed("table size");
  const lw_table* t = (const lw_table*)s.ptr[LW_SEC_TABLE];
  uint64_t kraft = 0; /* sum of 2^(11 - len) over coded symbols */
  for (int i = 0; i < t->alpha; ++i)
    if (t->code_len[i]) kraft += 1ull << (LW_MAX_CODE_LEN - t->code_len[i]);
  if (kraft != (1ull << LW_MAX_CODE_LEN) && !t->phantom) return failed("Kraft sum");
  if (s.bits_per_weight <= 0.0 || s.bits_per_weight >= 8.0) return failed("bits per weight");
  if (lw_validate_sections(&d, &s) != LW_OK) return failed("validate");

  const size_t n = lw_bundle_serialized_bytes(b);
  uint8_t* buf = (uint8_t*)malloc(n);
  if (!buf) return failed("malloc");
  if (lw_bundle_serialize(b, buf, n) != LW_OK) return failed("serialize");
  lw_bundle* c = NULL;
  if (lw_bundle_deserialize(buf, n, &c) != LW_OK || !c) return failed("deserialize");
  lw_sections s2;
  if (lw_bundle_sections(c, &s2) != LW_OK) return failed("sections of the copy");
  for (int i = 0; i < LW_NUM_SECTIONS; ++i) {
    if (s.bytes[i] != s2.bytes[i]) return failed("section size of the copy");
    if (s.bytes[i] && memcmp(s.ptr[i], s2.ptr[i], (size_t)s.bytes[i]) != 0)
      return failed("section bytes of the copy");
  }
  lw_desc d2;
  if (lw_bundle_desc(c, &d2) != LW_OK || d2.fmt != d.fmt || d2.rows != N || d2.cols != K)
    return failed("descriptor of the copy");

  buf[n / 2] ^= 0x40u; /* one flipped bit: the checksum must catch it */
  lw_bundle* bad = NULL;
  if (lw_bundle_deserialize(buf, n, &bad) != LW_ERR_CORRUPT || bad) return failed("corrupt copy");

  lw_desc odd = {LW_FMT_Q4_PAIR, 0, N + 1, K};
  if (lw_encode_bundle(&odd, codes, scales, mins, &bad) != LW_ERR_SHAPE) return failed("shape");
  if (lw_encode_bundle(&d, NULL, scales, mins, &bad) != LW_ERR_INVALID_ARG) return failed("NULL");
  if (lw_version() != 4) return failed("version");

  free(buf);
  lw_bundle_free(c);
  lw_bundle_free(b);
  printf("ok\n");
  return 0;
}
