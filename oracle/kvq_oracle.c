/*
 * kvq_oracle.c -- plain, slow, obviously-correct CPU oracle for the 2-bit paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library.  It shares no code, header, table or constant generator with the
 * CUDA path, and the CUDA path never calls it.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no FMA contraction, no fast-math), so every
 * float operation below is one IEEE-754 round-to-nearest-even operation in the written order.
 *
 * What it computes, and where the pages define it:
 *   - byte budget: "KV at 9 KB a token", section "How it works" (format table): a head's token
 *     costs 64 B of 2-bit code + an 8-byte metadata row = 72 B (BF16: 256 x 2 B = 512 B),
 *     x layers x KV heads x {K,V}; pages hold 64 tokens.
 *   - bytes per token formula: "Half the Cache, Twice the Context", section "Size the cache
 *     before you quantize it" (2 x layers x KV heads x head dim x bytes per value).
 *   - quantizer axes: same page, table "Two losses with one name" (scale K per channel,
 *     V per token -- the KIVI rule) and section "What the cache loses when you round it".
 *     The pages leave the 2-bit codebook open; the one fixed here is:
 *       V, per token, per 128-dim half: z = fp16(min), s = fp16((max-min)/3),
 *          c = clamp(rint((x - z)/s), 0, 3) (c = 0 when s == 0); v^ = z + c*s.
 *       K, per channel over a closed 64-token page: s_d = fp16(max|x|/3),
 *          c = clamp(rint((x/s_d + 3)/2), 0, 3) (c = 2 when s_d == 0); k^ = s_d*(2c-3).
 *     Keys of a page that is still open exist only in the exact BF16 ring ("the window of
 *     exact recent keys that the compressed KV format keeps": "The KV cache and prompt
 *     reuse", section "What a sequence is made of").
 *   - attention: softmax(sm_scale * q.k^) weighted sum of v^, in double precision, over the
 *     keys the page table addresses; prefill is causal (a query at position p sees t <= p).
 *   - rotated variant (format 2): the same 72 B rows over K and V rows rotated by the
 *     normalized 256-point Walsh-Hadamard transform before quantization (rotation named as
 *     what makes low-bit caches work in "Half the Cache, Twice the Context"); the ring keeps
 *     keys unrotated, dequantized page rows are turned back with H (H = H^T = H^-1).
 *   - per-token-K variant (format 3): the same 72 B rows, but each K row is quantized when it
 *     is appended, per token and per 128-dim half, by the V rule (z, s, c; k^ = z + c*s) --
 *     the axis that "Half the Cache, Twice the Context" ("What the cache loses when you round
 *     it", reading 1) finds better for K at 2 bits on its 3-level grid.  There is no page
 *     close; the ring still holds the last 64 keys exact, and a key is read from it only
 *     inside the window (t >= seq_len - window).
 *   - FP8 format (format 4): K and V rows stored as OCP FP8 E4M3 values (1 sign, 4 exponent
 *     bits with bias 7, 3 mantissa bits; no infinities; largest finite 448), one byte per value,
 *     256 B per head per token each -- half the bytes of BF16, the "2x capacity" FP8 cache of the
 *     vLLM study quoted in "Half the Cache, Twice the Context" ("What the vendors actually
 *     measured").  A per-tensor scale per K and V (geometry fields; 0 means 1) divides the
 *     input in fp32 before the conversion (round to nearest even, saturating at +-448) and
 *     multiplies the decoded value.  No ring: every key and value is read from its page.
 *   - accumulator model: "Half the Cache, Twice the Context", section "The cliff is in the
 *     accumulator, not the storage" (a running sum rounded after every add; two-level keeps
 *     an FP32 register).
 *
 * Rounding: every fp16/bf16 conversion here is written out from the IEEE-754 definition
 * (round to nearest, ties to even); rintf() is the C library's round-half-even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_D 256
#define ORC_P 64
#define ORC_FMT_HQ2B 0
#define ORC_FMT_BF16 1
#define ORC_FMT_HQ2B_HAD 2   /* the 2-bit format over Walsh-Hadamard-rotated K and V rows */
#define ORC_FMT_HQ2B_TOK 3   /* the 2-bit format with K quantized per token like V */
#define ORC_FMT_FP8 4        /* K and V rows as FP8 E4M3 with a per-tensor scale each */

/* status flags (same meaning as the device status word of the GPU library) */
#define ORC_PAGE_OOB 1
#define ORC_LEN_GT_TABLE 2
#define ORC_BAD_INPUT 4
#define ORC_BAD_LEN 8

typedef struct {
  int32_t format, num_layers, num_kv_heads, num_q_heads, head_dim, page_tokens;
  float k_scale, v_scale;   /* FP8 format only: per-tensor scales (0 means 1) */
} orc_geom;

/* ------------------------------------------------------------------ scalar conversions */
static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* float32 -> binary16, round to nearest, ties to even. */
uint16_t orc_f32_to_f16(float f) {
  uint32_t x = f32_bits(f);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax > 0x7F800000u) return sign | 0x7E00u;            /* NaN */
  if (ax == 0x7F800000u) return sign | 0x7C00u;           /* Inf */
  int bexp = (int)(ax >> 23);
  int e = bexp ? bexp - 127 : -126;                        /* unbiased exponent */
  uint32_t m = (ax & 0x7FFFFFu) | (bexp ? 0x800000u : 0u); /* value = m * 2^(e-23) */
  if (m == 0) return sign;
  /* quantum of the binary16 grid near this value: 2^(e-10) if normal, else 2^-24 */
  int qexp = e >= -14 ? e - 10 : -24;
  int shift = qexp - (e - 23);                            /* bits of m below the quantum */
  uint32_t r;
  if (shift >= 32) {
    r = 0;                                                 /* far below half a quantum */
  } else {
    r = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u))) r++;
  }
  if (e >= -14) {
    int E = e + 15;
    if (r == 0x800u) { r = 0x400u; E++; }                  /* mantissa carried out */
    if (E >= 31) return sign | 0x7C00u;                    /* overflow -> Inf */
    return (uint16_t)(sign | (uint32_t)(E << 10) | (r & 0x3FFu));
  }
  return (uint16_t)(sign | r);                             /* subnormal (r == 0x400 is 2^-14) */
}

float orc_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t E = (h >> 10) & 0x1Fu, M = h & 0x3FFu;
  if (E == 0x1Fu) return bits_f32(sign | 0x7F800000u | (M << 13));
  if (E == 0) {                                            /* zero / subnormal: M * 2^-24 */
    float v = (float)M * 5.9604644775390625e-08f;
    return sign ? -v : v;
  }
  return bits_f32(sign | ((E - 15 + 127) << 23) | (M << 13));
}

float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* float32 rounded to the nearest bfloat16 (ties to even), returned as float32. */
float orc_round_bf16(float f) {
  uint32_t u = f32_bits(f);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  return bits_f32(u);
}

/* ------------------------------------------------------------------ sizes */
/* 2 x layers x KV heads x head dim x bytes per value. */
double orc_kv_bytes_per_token(int layers, int kv_heads, int head_dim, double bytes_per_value) {
  return 2.0 * layers * kv_heads * head_dim * bytes_per_value;
}

/* bytes one head's one token costs for K or for V in each format */
int64_t orc_head_token_bytes(int format) {
  if (format == ORC_FMT_HQ2B || format == ORC_FMT_HQ2B_HAD || format == ORC_FMT_HQ2B_TOK)
    return 64 + 8;   /* 64 B code + 8 B meta row */
  if (format == ORC_FMT_BF16) return ORC_D * 2;
  if (format == ORC_FMT_FP8) return ORC_D;
  return -1;
}

int64_t orc_token_bytes(const orc_geom* g) {
  return (int64_t)g->num_layers * g->num_kv_heads * 2 * orc_head_token_bytes(g->format);
}

int64_t orc_page_bytes(const orc_geom* g) { return (int64_t)ORC_P * orc_token_bytes(g); }

/* bytes of one (layer, kv head, K-or-V) block of one page */
static int64_t block_bytes(const orc_geom* g) { return (int64_t)ORC_P * orc_head_token_bytes(g->format); }

/* byte offset of the (layer, head, kv) block inside a page: blocks are ordered
 * [layer][kv_head][K, V]. */
static int64_t block_offset(const orc_geom* g, int layer, int head, int kv) {
  return (((int64_t)layer * g->num_kv_heads + head) * 2 + kv) * block_bytes(g);
}

/* ------------------------------------------------------------------ quantizer */
static int input_ok(const uint16_t* x, int n) {
  for (int i = 0; i < n; i++) {
    float f = orc_bf16_to_f32(x[i]);
    if (!(fabsf(f) <= 65504.0f)) return 0;                 /* also rejects NaN / Inf */
  }
  return 1;
}

static float clamp03(float r) { return r < 0.0f ? 0.0f : (r > 3.0f ? 3.0f : r); }

/* V: one token row of one head (256 floats) -> 64 code bytes + meta row [s0, z0, s1, z1]. */
void orc_quant_v_row_f32(const float* x, uint8_t* codes, uint16_t* meta) {
  memset(codes, 0, 64);
  for (int half = 0; half < 2; half++) {
    int d0 = half * 128;
    float mn = x[d0], mx = mn;
    for (int d = d0; d < d0 + 128; d++) {
      float v = x[d];
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
    uint16_t z = orc_f32_to_f16(mn);
    float range = mx - mn;
    uint16_t s = orc_f32_to_f16(range / 3.0f);
    float zf = orc_f16_to_f32(z), sf = orc_f16_to_f32(s);
    for (int d = d0; d < d0 + 128; d++) {
      int c = 0;
      if (sf != 0.0f) {
        float diff = x[d] - zf;
        float t = diff / sf;
        c = (int)clamp03(rintf(t));
      }
      codes[d / 4] |= (uint8_t)(c << (2 * (d % 4)));
    }
    meta[2 * half] = s;
    meta[2 * half + 1] = z;
  }
}

/* V from bf16 (the plain format): the same steps on the exact float values. */
void orc_quant_v_row(const uint16_t* x, uint8_t* codes, uint16_t* meta) {
  float f[ORC_D];
  for (int d = 0; d < ORC_D; d++) f[d] = orc_bf16_to_f32(x[d]);
  orc_quant_v_row_f32(f, codes, meta);
}

/* K: one closed page of one head (64 rows x 256 floats) -> 64 x 64 code bytes + 256 scales. */
void orc_quant_k_page_f32(const float* x, uint8_t* codes, uint16_t* scales) {
  memset(codes, 0, 64 * 64);
  for (int d = 0; d < ORC_D; d++) {
    float a = 0.0f;
    for (int t = 0; t < ORC_P; t++) {
      float v = fabsf(x[t * ORC_D + d]);
      if (v > a) a = v;
    }
    uint16_t s = orc_f32_to_f16(a / 3.0f);
    float sf = orc_f16_to_f32(s);
    scales[d] = s;
    for (int t = 0; t < ORC_P; t++) {
      int c = 2;
      if (sf != 0.0f) {
        float u = x[t * ORC_D + d] / sf;
        u = u + 3.0f;
        u = 0.5f * u;
        c = (int)clamp03(rintf(u));
      }
      codes[t * 64 + d / 4] |= (uint8_t)(c << (2 * (d % 4)));
    }
  }
}

/* K from bf16 (the plain format). */
void orc_quant_k_page(const uint16_t* x, uint8_t* codes, uint16_t* scales) {
  float* f = (float*)malloc(sizeof(float) * ORC_P * ORC_D);
  for (int i = 0; i < ORC_P * ORC_D; i++) f[i] = orc_bf16_to_f32(x[i]);
  orc_quant_k_page_f32(f, codes, scales);
  free(f);
}

/* ------------------------------------------------------------------ Hadamard rotation
 * The rotated variant (a 256-point Walsh-Hadamard transform on K and V before 2-bit
 * quantization; "Half the Cache, Twice the Context" cites rotation as what makes low-bit
 * caches work): H = the Sylvester-ordered 256 x 256 Hadamard matrix / 16, so H = H^T = H^-1.
 * The quantizer's input is defined as the fast transform in float: stages h = 1, 2, 4, ..., 128,
 * each pair (i, i+h) -> (a + b, a - b) as one IEEE operation each, then x 1/16 (exact). */
void orc_fwht_f32(float* x) {
  for (int h = 1; h < ORC_D; h <<= 1)
    for (int i = 0; i < ORC_D; i += 2 * h)
      for (int j = i; j < i + h; j++) {
        float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
  for (int i = 0; i < ORC_D; i++) x[i] = x[i] * 0.0625f;
}

/* H x in double, written from the definition H[i][j] = (-1)^popcount(i & j) / 16. */
void orc_hadamard_f64(const double* x, double* y) {
  for (int i = 0; i < ORC_D; i++) {
    double acc = 0.0;
    for (int j = 0; j < ORC_D; j++) acc += (__builtin_popcount(i & j) & 1) ? -x[j] : x[j];
    y[i] = acc / 16.0;
  }
}

/* ------------------------------------------------------------------ FP8 E4M3
 * Encode a float as E4M3 by the format's definition: the representable magnitudes below 2^-6
 * are the multiples of 2^-9 (exponent field 0); from 2^e (e >= -6) up to 2^(e+1) they are the
 * multiples of 2^(e-3).  Round to the nearest multiple, ties to even; magnitudes past 448 give
 * 448 (saturation: the format has no infinity, and 464, the tie, also rounds to 448). */
uint8_t orc_f32_to_e4m3(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  int ex;
  frexp(a, &ex);                          /* a = f 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
  int e = a == 0.0 ? -6 : ex - 1;
  if (e < -6) e = -6;
  double quantum = ldexp(1.0, e - 3);
  double n = a / quantum;                 /* exact: a power-of-two scaling */
  double r = floor(n);
  double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double v = r * quantum;                 /* the rounded magnitude, at most 448 */
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)(v / ldexp(1.0, -9));             /* subnormal */
  frexp(v, &ex);
  int E = ex - 1 + 7;
  int m = (int)(v / ldexp(1.0, ex - 1) * 8.0) - 8;
  return sign | (uint8_t)(E << 3) | (uint8_t)m;
}

double orc_e4m3_to_f64(uint8_t b) {
  int E = (b >> 3) & 15, m = b & 7;
  double s = (b & 0x80) ? -1.0 : 1.0;
  if (E == 15 && m == 7) return NAN;
  if (E == 0) return s * m * ldexp(1.0, -9);
  return s * (1.0 + m / 8.0) * ldexp(1.0, E - 7);
}

static float fp8_scale(const orc_geom* g, int kv) {
  float s = kv ? g->v_scale : g->k_scale;
  return s == 0.0f ? 1.0f : s;
}

static int f32_ok(const float* x, int n) {
  for (int i = 0; i < n; i++)
    if (!(fabsf(x[i]) <= 65504.0f)) return 0;
  return 1;
}

static int code_at(const uint8_t* row, int d) { return (row[d / 4] >> (2 * (d % 4))) & 3; }

/* v^ = z + c*s per half, exact in double. */
void orc_dequant_v_row(const uint8_t* codes, const uint16_t* meta, double* out) {
  for (int d = 0; d < ORC_D; d++) {
    int half = d / 128;
    double s = orc_f16_to_f32(meta[2 * half]), z = orc_f16_to_f32(meta[2 * half + 1]);
    out[d] = z + code_at(codes, d) * s;
  }
}

/* k^ = s_d * (2c - 3), exact in double. */
void orc_dequant_k_row(const uint8_t* codes_row, const uint16_t* scales, double* out) {
  for (int d = 0; d < ORC_D; d++)
    out[d] = (double)orc_f16_to_f32(scales[d]) * (2 * code_at(codes_row, d) - 3);
}

/* ------------------------------------------------------------------ the paged cache */
static int geom_ok(const orc_geom* g) {
  if (g && g->format == ORC_FMT_FP8 &&
      (!(g->k_scale >= 0.0f && g->k_scale <= 3.0e38f) || !(g->v_scale >= 0.0f && g->v_scale <= 3.0e38f)))
    return 0;
  return g && (g->format == ORC_FMT_HQ2B || g->format == ORC_FMT_BF16 || g->format == ORC_FMT_HQ2B_HAD ||
               g->format == ORC_FMT_HQ2B_TOK || g->format == ORC_FMT_FP8) &&
         g->head_dim == ORC_D &&
         g->page_tokens == ORC_P && g->num_layers > 0 && g->num_kv_heads > 0 &&
         g->num_q_heads > 0 && g->num_q_heads % g->num_kv_heads == 0;
}

static uint16_t* ring_row(uint16_t* ring, const orc_geom* g, int lane, int layer, int head, int slot) {
  return ring + ((((int64_t)lane * g->num_layers + layer) * g->num_kv_heads + head) * ORC_P + slot) * ORC_D;
}

/*
 * Append n_new[b] tokens to every lane b, one token at a time in position order.  Token row
 * tok_offset[b]+i of k/v ([rows][Hkv][256] bf16) lands at position start_pos[b]+i.  In the
 * 2-bit format the V row is quantized at once; the K row goes to ring slot pos % 64, and when
 * slot 63 is written the page closes and its K block is quantized from the ring.  In the
 * per-token-K format the K row is quantized at once as well (V rule, into the K block's code and
 * meta rows) and also written to the ring; nothing happens at slot 63.  In the BF16 format both
 * rows are stored as they are.  Returns OR-ed status flags.
 */
int orc_append(const orc_geom* g, int layer, uint8_t* pool, int64_t pool_bytes, uint16_t* ring,
               const int32_t* page_table, int max_pages, int lanes, const int32_t* start_pos,
               const int32_t* n_new, const int32_t* tok_offset, const uint16_t* k, const uint16_t* v) {
  if (!geom_ok(g) || layer < 0 || layer >= g->num_layers) return -1;
  int status = 0;
  int64_t pb = orc_page_bytes(g);
  int64_t npages = pool_bytes / pb;
  int H = g->num_kv_heads;
  for (int b = 0; b < lanes; b++) {
    for (int i = 0; i < n_new[b]; i++) {
      int64_t t = (int64_t)start_pos[b] + i;
      int64_t row = (int64_t)tok_offset[b] + i;
      if (t / ORC_P >= max_pages) { status |= ORC_LEN_GT_TABLE; continue; }
      int32_t phys = page_table[(int64_t)b * max_pages + t / ORC_P];
      if (phys < 0 || phys >= npages) { status |= ORC_PAGE_OOB; continue; }
      int slot = (int)(t % ORC_P);
      uint8_t* page = pool + (int64_t)phys * pb;
      for (int h = 0; h < H; h++) {
        const uint16_t* kx = k + (row * H + h) * ORC_D;
        const uint16_t* vx = v + (row * H + h) * ORC_D;
        if (!input_ok(kx, ORC_D) || !input_ok(vx, ORC_D)) { status |= ORC_BAD_INPUT; continue; }
        uint8_t* kblk = page + block_offset(g, layer, h, 0);
        uint8_t* vblk = page + block_offset(g, layer, h, 1);
        if (g->format == ORC_FMT_BF16) {
          memcpy(kblk + (int64_t)slot * ORC_D * 2, kx, ORC_D * 2);
          memcpy(vblk + (int64_t)slot * ORC_D * 2, vx, ORC_D * 2);
          continue;
        }
        if (g->format == ORC_FMT_FP8) {   /* x / scale in fp32, then E4M3 */
          float ks = fp8_scale(g, 0), vs = fp8_scale(g, 1);
          for (int d = 0; d < ORC_D; d++) {
            kblk[(int64_t)slot * ORC_D + d] = orc_f32_to_e4m3(orc_bf16_to_f32(kx[d]) / ks);
            vblk[(int64_t)slot * ORC_D + d] = orc_f32_to_e4m3(orc_bf16_to_f32(vx[d]) / vs);
          }
          continue;
        }
        uint16_t meta[4];
        if (g->format == ORC_FMT_HQ2B_HAD) {
          /* the rotated V row is quantized; the ring keeps the key as it came (exact) */
          float f[ORC_D];
          for (int d = 0; d < ORC_D; d++) f[d] = orc_bf16_to_f32(vx[d]);
          orc_fwht_f32(f);
          if (!f32_ok(f, ORC_D)) { status |= ORC_BAD_INPUT; continue; }
          orc_quant_v_row_f32(f, vblk + slot * 64, meta);
        } else {
          orc_quant_v_row(vx, vblk + slot * 64, meta);
        }
        memcpy(vblk + 4096 + slot * 8, meta, 8);
        memcpy(ring_row(ring, g, b, layer, h, slot), kx, ORC_D * 2);
        if (g->format == ORC_FMT_HQ2B_TOK) {
          /* the key row is quantized now, by the V rule, into the K block's own rows */
          orc_quant_v_row(kx, kblk + slot * 64, meta);
          memcpy(kblk + 4096 + slot * 8, meta, 8);
        } else if (slot == ORC_P - 1) {
          uint16_t scales[ORC_D];
          if (g->format == ORC_FMT_HQ2B_HAD) {
            /* the page's 64 keys, each rotated, quantized per channel of the rotated basis */
            float* f = (float*)malloc(sizeof(float) * ORC_P * ORC_D);
            const uint16_t* r0 = ring_row(ring, g, b, layer, h, 0);
            for (int i = 0; i < ORC_P * ORC_D; i++) f[i] = orc_bf16_to_f32(r0[i]);
            int ok = 1;
            for (int t2 = 0; t2 < ORC_P; t2++) {
              orc_fwht_f32(f + t2 * ORC_D);
              ok = ok && f32_ok(f + t2 * ORC_D, ORC_D);
            }
            if (ok) {
              orc_quant_k_page_f32(f, kblk, scales);
              memcpy(kblk + 4096, scales, sizeof scales);
            } else {
              status |= ORC_BAD_INPUT;
            }
            free(f);
          } else {
            orc_quant_k_page(ring_row(ring, g, b, layer, h, 0), kblk, scales);
            memcpy(kblk + 4096, scales, sizeof scales);
          }
        }
      }
    }
  }
  return status;
}

/* The key of position t as the attention sees it (double), given the lane's cache state of
 * seq_len tokens: in the 2-bit formats keys at t >= min(seq_len - window, first position of
 * the open page) come from the exact ring (per-token-K format: t >= seq_len - window), the
 * rest are dequantized from their page. */
static int load_key(const orc_geom* g, int layer, const uint8_t* pool, int64_t npages,
                    const uint16_t* ring, int window, const int32_t* page_row, int max_pages,
                    int lane, int seq_len, int head, int64_t t, double* out) {
  int64_t open_start = (int64_t)(seq_len / ORC_P) * ORC_P;
  int64_t exact_from = seq_len - window < open_start ? seq_len - window : open_start;
  if (g->format == ORC_FMT_HQ2B_TOK) exact_from = seq_len - window;   /* every key has codes */
  if (g->format != ORC_FMT_BF16 && g->format != ORC_FMT_FP8 && t >= exact_from) {
    const uint16_t* r = ring_row((uint16_t*)ring, g, lane, layer, head, (int)(t % ORC_P));
    for (int d = 0; d < ORC_D; d++) out[d] = orc_bf16_to_f32(r[d]);
    return 0;
  }
  if (t / ORC_P >= max_pages) return ORC_LEN_GT_TABLE;
  int32_t phys = page_row[t / ORC_P];
  if (phys < 0 || phys >= npages) return ORC_PAGE_OOB;
  const uint8_t* blk = pool + (int64_t)phys * orc_page_bytes(g) + block_offset(g, layer, head, 0);
  int slot = (int)(t % ORC_P);
  if (g->format == ORC_FMT_BF16) {
    const uint16_t* r = (const uint16_t*)(blk + (int64_t)slot * ORC_D * 2);
    for (int d = 0; d < ORC_D; d++) out[d] = orc_bf16_to_f32(r[d]);
  } else if (g->format == ORC_FMT_FP8) {
    for (int d = 0; d < ORC_D; d++) out[d] = orc_e4m3_to_f64(blk[(int64_t)slot * ORC_D + d]) * fp8_scale(g, 0);
  } else if (g->format == ORC_FMT_HQ2B_TOK) {
    orc_dequant_v_row(blk + slot * 64, (const uint16_t*)(blk + 4096 + slot * 8), out);
  } else {
    orc_dequant_k_row(blk + slot * 64, (const uint16_t*)(blk + 4096), out);
    if (g->format == ORC_FMT_HQ2B_HAD) {   /* the page holds H k: k^ = H (H k)^ */
      double r[ORC_D];
      orc_hadamard_f64(out, r);
      memcpy(out, r, sizeof r);
    }
  }
  return 0;
}

static int load_value(const orc_geom* g, int layer, const uint8_t* pool, int64_t npages,
                      const int32_t* page_row, int max_pages, int head, int64_t t, double* out) {
  if (t / ORC_P >= max_pages) return ORC_LEN_GT_TABLE;
  int32_t phys = page_row[t / ORC_P];
  if (phys < 0 || phys >= npages) return ORC_PAGE_OOB;
  const uint8_t* blk = pool + (int64_t)phys * orc_page_bytes(g) + block_offset(g, layer, head, 1);
  int slot = (int)(t % ORC_P);
  if (g->format == ORC_FMT_BF16) {
    const uint16_t* r = (const uint16_t*)(blk + (int64_t)slot * ORC_D * 2);
    for (int d = 0; d < ORC_D; d++) out[d] = orc_bf16_to_f32(r[d]);
  } else if (g->format == ORC_FMT_FP8) {
    for (int d = 0; d < ORC_D; d++) out[d] = orc_e4m3_to_f64(blk[(int64_t)slot * ORC_D + d]) * fp8_scale(g, 1);
  } else {
    orc_dequant_v_row(blk + slot * 64, (const uint16_t*)(blk + 4096 + slot * 8), out);
    if (g->format == ORC_FMT_HQ2B_HAD) {   /* the page holds H v: v^ = H (H v)^ */
      double r[ORC_D];
      orc_hadamard_f64(out, r);
      memcpy(out, r, sizeof r);
    }
  }
  return 0;
}

/*
 * One query row of query head q_head of lane `lane` attends keys 0 .. n_keys-1:
 *   s_t = sm_scale * sum_d q_d k^_{t,d};  out = sum_t exp(s_t - max) v^_t / sum_t exp(s_t - max)
 * in double.  The query head reads KV head q_head / (Hq / Hkv) (contiguous GQA groups).
 * n_keys == 0 gives out = 0.  *top1 (if not NULL) receives the index of the largest score
 * (first one on ties).  Returns status flags.
 */
int orc_attend(const orc_geom* g, int layer, const uint8_t* pool, int64_t pool_bytes,
               const uint16_t* ring, int window, const int32_t* page_row, int max_pages, int lane,
               int seq_len, int q_head, const uint16_t* q_row, int64_t n_keys, double sm_scale,
               double* out, int64_t* top1) {
  if (!geom_ok(g)) return -1;
  int64_t npages = pool_bytes / orc_page_bytes(g);
  int head = q_head / (g->num_q_heads / g->num_kv_heads);
  double q[ORC_D], kv[ORC_D];
  for (int d = 0; d < ORC_D; d++) q[d] = orc_bf16_to_f32(q_row[d]);
  for (int d = 0; d < ORC_D; d++) out[d] = 0.0;
  if (top1) *top1 = -1;
  if (n_keys <= 0) return 0;
  double* s = (double*)malloc(sizeof(double) * (size_t)n_keys);
  if (!s) return -1;
  int status = 0;
  double mx = -INFINITY;
  for (int64_t t = 0; t < n_keys; t++) {
    int st = load_key(g, layer, pool, npages, ring, window, page_row, max_pages, lane, seq_len, head, t, kv);
    if (st) { status |= st; s[t] = -INFINITY; continue; }
    double dot = 0.0;
    for (int d = 0; d < ORC_D; d++) dot += q[d] * kv[d];
    s[t] = sm_scale * dot;
    if (s[t] > mx) { mx = s[t]; if (top1) *top1 = t; }
  }
  double den = 0.0;
  for (int64_t t = 0; t < n_keys; t++) {
    if (s[t] == -INFINITY) continue;
    double w = exp(s[t] - mx);
    int st = load_value(g, layer, pool, npages, page_row, max_pages, head, t, kv);
    if (st) { status |= st; continue; }
    den += w;
    for (int d = 0; d < ORC_D; d++) out[d] += w * kv[d];
  }
  if (den > 0.0)
    for (int d = 0; d < ORC_D; d++) out[d] /= den;
  free(s);
  return status;
}

/* Decode: for every lane b and query head j, q[b][j] (bf16 [lanes][Hq][256]) attends all
 * seq_len[b] keys; out is double [lanes][Hq][256]. */
int orc_decode(const orc_geom* g, int layer, const uint8_t* pool, int64_t pool_bytes,
               const uint16_t* ring, int window, const int32_t* page_table, int max_pages, int lanes,
               const int32_t* seq_len, const uint16_t* q, double sm_scale, double* out) {
  int status = 0, Hq = g->num_q_heads;
  for (int b = 0; b < lanes; b++)
    for (int j = 0; j < Hq; j++) {
      int st = orc_attend(g, layer, pool, pool_bytes, ring, window, page_table + (int64_t)b * max_pages,
                          max_pages, b, seq_len[b], j, q + ((int64_t)b * Hq + j) * ORC_D, seq_len[b],
                          sm_scale, out + ((int64_t)b * Hq + j) * ORC_D, NULL);
      if (st < 0) return st;
      status |= st;
    }
  return status;
}

/* Prefill: lane b's query rows q_offset[b] .. q_offset[b]+n_q[b]-1 (bf16 [rows][Hq][256]) sit
 * at positions q_pos0[b] + i and attend causally to keys 0 .. q_pos0[b]+i; out is double
 * [rows][Hq][256]. */
int orc_prefill(const orc_geom* g, int layer, const uint8_t* pool, int64_t pool_bytes,
                const uint16_t* ring, int window, const int32_t* page_table, int max_pages, int lanes,
                const int32_t* q_pos0, const int32_t* n_q, const int32_t* q_offset,
                const int32_t* seq_len, const uint16_t* q, double sm_scale, double* out) {
  int status = 0, Hq = g->num_q_heads;
  for (int b = 0; b < lanes; b++)
    for (int i = 0; i < n_q[b]; i++) {
      int64_t pos = (int64_t)q_pos0[b] + i, row = (int64_t)q_offset[b] + i;
      if (pos >= seq_len[b]) { status |= ORC_BAD_LEN; continue; }
      for (int j = 0; j < Hq; j++) {
        int st = orc_attend(g, layer, pool, pool_bytes, ring, window, page_table + (int64_t)b * max_pages,
                            max_pages, b, seq_len[b], j, q + (row * Hq + j) * ORC_D, pos + 1, sm_scale,
                            out + (row * Hq + j) * ORC_D, NULL);
        if (st < 0) return st;
        status |= st;
      }
    }
  return status;
}

/* ------------------------------------------------------------------ accumulator model */
/* Round x to the precision a running accumulator keeps: kind 0 = fp32, 1 = fp16, 2 = bf16. */
static double round_acc(double x, int kind) {
  float f = (float)x;
  if (kind == 0) return f;
  if (kind == 1) return orc_f16_to_f32(orc_f32_to_f16(f));
  return orc_round_bf16(f);
}

/* Sum n equal weights 1/n in a running accumulator rounded after every add (flat), or, with
 * two_level, in an FP32 register rounded to the storage type once at the end. */
double orc_flat_sum(int n, int kind, int two_level) {
  double term = 1.0 / n, acc = 0.0;
  for (int i = 0; i < n; i++) acc = two_level ? (double)(float)(acc + term) : round_acc(acc + term, kind);
  return two_level ? round_acc(acc, kind) : acc;
}
