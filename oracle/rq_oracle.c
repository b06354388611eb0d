/*
 * rq_oracle.c -- plain, slow, fp64 CPU oracle for the rotation-quantized KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in __graft_entry__.py and the
 * cpu_baseline leg of bench.py may load this file's library.  The CUDA library never links,
 * includes or calls it, and this file includes nothing from the CUDA library.
 *
 * What it follows ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache Compression";
 * section "TurboQuant KV Cache Compression"; "Acknowledgments"):
 *   - RotorQuant modes rq3/rq4 x planar/iso: 2D Givens rotations (PlanarQuant) or 4D
 *     quaternion rotations (IsoQuant), data-oblivious, then low-bit scalar codes;
 *   - rotation cost per 128-d vector: 256 FMAs planar, 512 iso, 16,384 for a dense rotation;
 *   - the scalar quantizer is Lloyd-Max (credited to TurboQuant: random rotation + Lloyd-Max
 *     scalar quantization).
 * The pages do not fix norm handling, codebook scaling, pairing, bit layout, page layout or
 * attention; the reading taken for each is stated at the function that uses it.
 *
 * Everything is computed in double precision, one vector or one (sequence, head) at a time,
 * with no blocking or fusion.  The one decision taken in single precision is the scalar code:
 * u = y/n is rounded to float and compared with the float bin boundaries, which is the
 * precision the GPU kernel decides in.
 *
 * Parity pins (tests/test_oracle_*.py): fp16 rounding against numpy; Lloyd-Max against the
 * 2-level closed form, Max (1960) Table I and numerical quadrature; rotations against
 * quaternion-as-complex-matrix products, materialised matrices and the FMA counts above;
 * coding against brute-force nearest centroid; packing against hand-written fixtures;
 * attention against torch's scaled_dot_product_attention and closed-form special cases.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>

/* ------------------------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> double, written from the format's definition.                   */
/* ------------------------------------------------------------------------------------- */

double rqo_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exp = (h >> 10) & 0x1f;
  int man = h & 0x3ff;
  double v;
  if (exp == 0) {
    v = ldexp((double)man, -24);                  /* subnormal: man * 2^-14 * 2^-10 */
  } else if (exp == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + man), exp - 25);    /* (1 + man/1024) * 2^(exp-15) */
  }
  return sign ? -v : v;
}

/* Round to nearest, ties to even; overflow goes to infinity. */
uint16_t rqo_double_to_half(double x) {
  uint16_t sign = 0;
  if (isnan(x)) return 0x7e00;
  if (signbit(x)) { sign = 0x8000; x = -x; }
  if (x == 0.0) return sign;
  if (x >= 65520.0) return sign | 0x7c00;       /* 65520 = max finite + half an ulp */
  int e;
  frexp(x, &e);                                  /* x = f * 2^e, f in [0.5, 1) */
  int exp16 = e - 1 + 15;                        /* biased exponent of x = 1.m * 2^(e-1) */
  double scaled;
  if (exp16 <= 0) {
    scaled = ldexp(x, 24);                       /* subnormal grid: units of 2^-24 */
  } else {
    scaled = ldexp(x, 10 - (e - 1));             /* units of 2^(e-1-10): [1024, 2048) */
  }
  double fl = floor(scaled);
  double rem = scaled - fl;
  uint32_t q = (uint32_t)fl;
  if (rem > 0.5 || (rem == 0.5 && (q & 1))) q += 1;
  if (exp16 <= 0) {
    return sign | (uint16_t)q;                   /* q may reach 1024 = smallest normal */
  }
  if (q == 2048) { q = 1024; exp16 += 1; }
  if (exp16 >= 31) return sign | 0x7c00;
  return sign | (uint16_t)((exp16 << 10) | (q - 1024));
}

/* ------------------------------------------------------------------------------------- */
/* Lloyd-Max quantizer for the standard normal (the scalar quantizer of the method).      */
/* Condition 1: each threshold is the midpoint of its two neighbouring levels.            */
/* Condition 2: each level is the conditional mean of N(0,1) over its cell.               */
/* Iterated from a uniform start until the levels stop moving.                            */
/* ------------------------------------------------------------------------------------- */

static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }

/* P(a < X <= b) for X ~ N(0,1), computed from erfc on the side that avoids cancellation. */
static double normal_mass(double a, double b) {
  const double r = 1.0 / sqrt(2.0);
  if (a >= 0.0) return 0.5 * (erfc(a * r) - erfc(b * r));
  if (b <= 0.0) return 0.5 * (erfc(-b * r) - erfc(-a * r));
  return 0.5 * (erf(b * r) - erf(a * r));
}

static double bphi(double x) { return isinf(x) ? 0.0 : x * phi(x); }

/* Fills c[levels] (ascending) and t[levels-1]; returns the iteration count. */
int rqo_lloyd_max_normal(int levels, double *c, double *t, double *mse) {
  if (levels < 2 || levels > 256) return -1;
  for (int j = 0; j < levels; ++j) c[j] = -3.0 + 6.0 * (j + 0.5) / levels;
  int it;
  for (it = 1; it <= 2000000; ++it) {
    for (int j = 0; j + 1 < levels; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
    double moved = 0.0;
    for (int j = 0; j < levels; ++j) {
      double a = (j == 0) ? -INFINITY : t[j - 1];
      double b = (j == levels - 1) ? INFINITY : t[j];
      double pa = isinf(a) ? 0.0 : phi(a);
      double pb = isinf(b) ? 0.0 : phi(b);
      double cj = (pa - pb) / normal_mass(a, b);
      double dlt = fabs(cj - c[j]);
      if (dlt > moved) moved = dlt;
      c[j] = cj;
    }
    if (moved < 1e-15) break;
  }
  for (int j = 0; j + 1 < levels; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
  if (mse) {
    /* sum over cells of  E[(X - c_j)^2 ; cell j]  using
       int x^2 phi = [Phi - x phi],  int x phi = [-phi]. */
    double total = 0.0;
    for (int j = 0; j < levels; ++j) {
      double a = (j == 0) ? -INFINITY : t[j - 1];
      double b = (j == levels - 1) ? INFINITY : t[j];
      double pa = isinf(a) ? 0.0 : phi(a);
      double pb = isinf(b) ? 0.0 : phi(b);
      double p = normal_mass(a, b);
      double ex2 = p - (bphi(b) - bphi(a));
      double ex = pa - pb;
      total += ex2 - 2.0 * c[j] * ex + c[j] * c[j] * p;
    }
    *mse = total;
  }
  return it;
}

/* Codebook for the unit-norm rotated coordinates, which are close to N(0, 1/d):
   centroid_j = float(c_j / sqrt(d)),  boundary_j = float((centroid_j + centroid_{j+1}) / 2)
   with the midpoint taken in double from the float centroids. */
void rqo_codebook(int bits, int d, float *centroids, float *boundaries) {
  int levels = 1 << bits;
  double c[256], t[256];
  rqo_lloyd_max_normal(levels, c, t, NULL);
  double s = 1.0 / sqrt((double)d);
  for (int j = 0; j < levels; ++j) centroids[j] = (float)(c[j] * s);
  for (int j = 0; j + 1 < levels; ++j)
    boundaries[j] = (float)(0.5 * ((double)centroids[j] + (double)centroids[j + 1]));
}

/* ------------------------------------------------------------------------------------- */
/* Rotations.                                                                              */
/*   planar (PlanarQuant, 2D Givens): params [d/2][2] = (cos t, sin t) for pair (2i,2i+1):  */
/*       y_2i = cos*x_2i - sin*x_2i+1,   y_2i+1 = sin*x_2i + cos*x_2i+1                     */
/*   iso (IsoQuant, 4D quaternion): params [d/4][4] = unit quaternion (a,b,c,d) for block    */
/*       4i..4i+3, y_blk = q (x) x_blk, the Hamilton product with q on the left.            */
/*   dense (TurboQuant, "TurboQuant KV Cache Compression" section and "Acknowledgments":    */
/*       random rotation): params [d][d] = an orthogonal matrix R, row-major, y = R x.       */
/* The inverse applies the transpose.  Each returns the number of multiply-adds it made.    */
/* ------------------------------------------------------------------------------------- */

static void quat_left_matrix(const float *q, double L[4][4]) {
  double a = q[0], b = q[1], c = q[2], d = q[3];
  L[0][0] = a;  L[0][1] = -b; L[0][2] = -c; L[0][3] = -d;
  L[1][0] = b;  L[1][1] = a;  L[1][2] = -d; L[1][3] = c;
  L[2][0] = c;  L[2][1] = d;  L[2][2] = a;  L[2][3] = -b;
  L[3][0] = d;  L[3][1] = -c; L[3][2] = b;  L[3][3] = a;
}

long rqo_rotate(int mode, const float *params, int d, const double *x, double *y, int inverse) {
  long fma = 0;
  if (mode == 2) {
    for (int r = 0; r < d; ++r) {
      double acc = 0.0;
      for (int k = 0; k < d; ++k) {
        acc += (double)(inverse ? params[(size_t)k * d + r] : params[(size_t)r * d + k]) * x[k];
        fma += 1;
      }
      y[r] = acc;
    }
    return fma;
  }
  if (mode == 0) {
    for (int i = 0; i < d / 2; ++i) {
      double c = params[2 * i], s = params[2 * i + 1];
      double x0 = x[2 * i], x1 = x[2 * i + 1];
      if (!inverse) {
        y[2 * i] = c * x0 - s * x1;
        y[2 * i + 1] = s * x0 + c * x1;
      } else {
        y[2 * i] = c * x0 + s * x1;
        y[2 * i + 1] = -s * x0 + c * x1;
      }
      fma += 4;
    }
  } else {
    for (int blk = 0; blk < d / 4; ++blk) {
      double L[4][4];
      quat_left_matrix(params + 4 * blk, L);
      const double *xb = x + 4 * blk;
      double out[4];
      for (int r = 0; r < 4; ++r) {
        double acc = 0.0;
        for (int k = 0; k < 4; ++k) {
          acc += (inverse ? L[k][r] : L[r][k]) * xb[k];
          fma += 1;
        }
        out[r] = acc;
      }
      for (int r = 0; r < 4; ++r) y[4 * blk + r] = out[r];
    }
  }
  return fma;
}

/* The same rotation as a dense d x d matrix R (row-major), y = R x. */
void rqo_rotation_matrix(int mode, const float *params, int d, double *R) {
  for (int i = 0; i < d * d; ++i) R[i] = (mode == 2) ? (double)params[i] : 0.0;
  if (mode == 2) return;
  if (mode == 0) {
    for (int i = 0; i < d / 2; ++i) {
      double c = params[2 * i], s = params[2 * i + 1];
      R[(2 * i) * d + 2 * i] = c;       R[(2 * i) * d + 2 * i + 1] = -s;
      R[(2 * i + 1) * d + 2 * i] = s;   R[(2 * i + 1) * d + 2 * i + 1] = c;
    }
  } else {
    for (int blk = 0; blk < d / 4; ++blk) {
      double L[4][4];
      quat_left_matrix(params + 4 * blk, L);
      for (int r = 0; r < 4; ++r)
        for (int k = 0; k < 4; ++k) R[(4 * blk + r) * d + 4 * blk + k] = L[r][k];
    }
  }
}

/* Dense matrix-vector product (the cost of a dense rotation); transpose selects R^T. */
long rqo_matvec(const double *R, int d, const double *x, double *y, int transpose) {
  long fma = 0;
  for (int r = 0; r < d; ++r) {
    double acc = 0.0;
    for (int k = 0; k < d; ++k) {
      acc += (transpose ? R[k * d + r] : R[r * d + k]) * x[k];
      fma += 1;
    }
    y[r] = acc;
  }
  return fma;
}

/* ------------------------------------------------------------------------------------- */
/* Encoding of one vector.                                                                 */
/*   n = ||x|| (double), stored as n16 = fp16(n) rounded to nearest even;                  */
/*   y = R x;  u = y / n  (u = 0 when n = 0);                                              */
/*   code_i = #{ j : boundary_j < float(u_i) }  (a value on a boundary takes the lower bin); */
/*   margin_i = min_j |u_i - boundary_j|, the distance to the nearest boundary.             */
/* ------------------------------------------------------------------------------------- */

void rqo_encode(int mode, int bits, int d, const float *rot, const float *boundaries,
                const uint16_t *x16, uint8_t *codes, uint16_t *n16, double *margin) {
  int levels = 1 << bits;
  double x[1024], y[1024];
  double ss = 0.0;
  for (int i = 0; i < d; ++i) {
    x[i] = rqo_half_to_double(x16[i]);
    ss += x[i] * x[i];
  }
  double n = sqrt(ss);
  *n16 = rqo_double_to_half(n);
  rqo_rotate(mode, rot, d, x, y, 0);
  for (int i = 0; i < d; ++i) {
    double u = (n > 0.0) ? y[i] / n : 0.0;
    float uf = (float)u;
    int code = 0;
    double m = INFINITY;
    for (int j = 0; j + 1 < levels; ++j) {
      if (boundaries[j] < uf) code += 1;
      double dist = fabs(u - (double)boundaries[j]);
      if (dist < m) m = dist;
    }
    codes[i] = (uint8_t)code;
    if (margin) margin[i] = m;
  }
}

/* ------------------------------------------------------------------------------------- */
/* Bit layout of one vector's codes (the library's storage contract; the pages fix none).  */
/*   4-bit: byte j = code[2j] | code[2j+1] << 4                     (64 bytes for d = 128)  */
/*   3-bit: per 32-dim group w, 12 bytes at 12w = three little-endian words W0, W1, W2:     */
/*     W0 bits 2i..2i+1 = code[32w+i] & 3        (i = 0..15)                                */
/*     W1 bits 2i..2i+1 = code[32w+16+i] & 3     (i = 0..15)                                */
/*     W2 bit p(i)      = code[32w+i] >> 2       (i = 0..31), with i = 16h + 4k + r and     */
/*                        p(i) = 8k + 2h + {4, 5, 0, 1}[r]                                  */
/* ------------------------------------------------------------------------------------- */

static int hi_bit_pos(int i) {
  static const int off[4] = {4, 5, 0, 1};
  int h = i / 16, k = (i % 16) / 4, r = i % 4;
  return 8 * k + 2 * h + off[r];
}

size_t rqo_vector_bytes(int bits, int d) { return (size_t)d * bits / 8; }

static void put_word(uint8_t *p, uint32_t w) {
  for (int b = 0; b < 4; ++b) p[b] = (uint8_t)(w >> (8 * b));
}
static uint32_t get_word(const uint8_t *p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

void rqo_pack(int bits, int d, const uint8_t *codes, uint8_t *out) {
  if (bits == 2) {
    for (int j = 0; j < d / 4; ++j)
      out[j] = (uint8_t)((codes[4 * j] & 3) | ((codes[4 * j + 1] & 3) << 2) | ((codes[4 * j + 2] & 3) << 4) |
                         ((codes[4 * j + 3] & 3) << 6));
  } else if (bits == 4) {
    for (int j = 0; j < d / 2; ++j) out[j] = (uint8_t)((codes[2 * j] & 15) | ((codes[2 * j + 1] & 15) << 4));
  } else {
    for (int w = 0; w < d / 32; ++w) {
      const uint8_t *c = codes + 32 * w;
      uint32_t w0 = 0, w1 = 0, w2 = 0;
      for (int i = 0; i < 16; ++i) {
        w0 |= (uint32_t)(c[i] & 3) << (2 * i);
        w1 |= (uint32_t)(c[16 + i] & 3) << (2 * i);
      }
      for (int i = 0; i < 32; ++i) w2 |= (uint32_t)((c[i] >> 2) & 1) << hi_bit_pos(i);
      put_word(out + 12 * w, w0);
      put_word(out + 12 * w + 4, w1);
      put_word(out + 12 * w + 8, w2);
    }
  }
}

void rqo_unpack(int bits, int d, const uint8_t *in, uint8_t *codes) {
  if (bits == 2) {
    for (int j = 0; j < d / 4; ++j)
      for (int r = 0; r < 4; ++r) codes[4 * j + r] = (in[j] >> (2 * r)) & 3;
  } else if (bits == 4) {
    for (int j = 0; j < d / 2; ++j) {
      codes[2 * j] = in[j] & 15;
      codes[2 * j + 1] = in[j] >> 4;
    }
  } else {
    for (int w = 0; w < d / 32; ++w) {
      uint32_t w0 = get_word(in + 12 * w), w1 = get_word(in + 12 * w + 4), w2 = get_word(in + 12 * w + 8);
      for (int i = 0; i < 32; ++i) {
        uint32_t lo = (i < 16) ? (w0 >> (2 * i)) & 3 : (w1 >> (2 * (i - 16))) & 3;
        uint32_t hi = (w2 >> hi_bit_pos(i)) & 1;
        codes[32 * w + i] = (uint8_t)(lo | (hi << 2));
      }
    }
  }
}

/* x_hat = n16 * R^T c[code] */
void rqo_dequant(int mode, int bits, int d, const float *rot, const float *centroids,
                 const uint8_t *codes, uint16_t n16, double *xhat) {
  (void)bits;
  double y[1024];
  double n = rqo_half_to_double(n16);
  for (int i = 0; i < d; ++i) y[i] = (double)centroids[codes[i]];
  rqo_rotate(mode, rot, d, y, xhat, 1);
  for (int i = 0; i < d; ++i) xhat[i] *= n;
}

/* ------------------------------------------------------------------------------------- */
/* Paged cache.  One chunk per (page, kv head), at byte (page * Hkv + head) * page_bytes:   */
/*   K codes [P][vb] | V codes [P][vb] | K norms fp16 [P] | V norms fp16 [P]               */
/* with vb = d * bits / 8.  Slot s holds token offset s % P of page s / P.                 */
/* K codes, and 3-bit V codes, are stored token after token, in units of 8 bytes.  4-bit   */
/* and 2-bit V codes (d = 128) are stored as token pairs, in units of one 16-dim group      */
/* (8 bytes at 4 bits, 4 bytes at 2 bits): pair p = tokens (2p, 2p+1) fills 2 * vb bytes,  */
/* and the unit of group c of token 2p + h sits at byte                                     */
/*   4-bit:  16 * (c ^ (2p mod 8)) + 8h                                                     */
/*   2-bit:   8 * (c ^ (4 * ((p >> 1) & 1))) + 4h                                           */
/* of the pair.                                                                             */
/* ------------------------------------------------------------------------------------- */

static int v_unit_bytes(int bits, int d) { return ((bits == 4 || bits == 2) && d == 128) ? 2 * bits : 8; }

/* Byte offset, inside the V-codes section, of unit `unit` of token `off`. */
static size_t v_unit_offset(int bits, int d, int off, int unit) {
  size_t vb = rqo_vector_bytes(bits, d);
  if (d != 128 || bits == 3) return (size_t)off * vb + (size_t)unit * 8;
  int pair = off / 2, h = off % 2;
  if (bits == 4) return (size_t)pair * 128 + (size_t)16 * (unit ^ ((2 * pair) % 8)) + (size_t)8 * h;
  return (size_t)pair * 64 + (size_t)8 * (unit ^ (4 * ((pair >> 1) & 1))) + (size_t)4 * h;
}

static void put_v(int bits, int d, uint8_t *vsec, int off, const uint8_t *packed) {
  size_t vb = rqo_vector_bytes(bits, d);
  int ub = v_unit_bytes(bits, d);
  for (size_t u = 0; u < vb / ub; ++u) memcpy(vsec + v_unit_offset(bits, d, off, (int)u), packed + ub * u, ub);
}

static void get_v(int bits, int d, const uint8_t *vsec, int off, uint8_t *packed) {
  size_t vb = rqo_vector_bytes(bits, d);
  int ub = v_unit_bytes(bits, d);
  for (size_t u = 0; u < vb / ub; ++u) memcpy(packed + ub * u, vsec + v_unit_offset(bits, d, off, (int)u), ub);
}

/* Exposed for tests: byte offset of unit `unit` of V token `off` in its section, and the
   unit size in bytes. */
size_t rqo_v_unit_offset(int bits, int d, int off, int unit) { return v_unit_offset(bits, d, off, unit); }
int rqo_v_unit_bytes(int bits, int d) { return v_unit_bytes(bits, d); }

/* Floats of one head's rotation parameters: d for planar / iso, d * d for dense. */
static size_t rot_stride(int mode, int d) { return mode == 2 ? (size_t)d * d : (size_t)d; }

size_t rqo_page_bytes(int bits, int page_size, int d) {
  return (size_t)page_size * (2 * rqo_vector_bytes(bits, d) + 4);
}

/* k, v: fp16 [n][Hkv][d].  Slots < 0 are skipped.  margin_k / margin_v (nullable): [n][Hkv][d]. */
void rqo_append(int mode, int bits, int d, int hkv, int page_size,
                const float *rot_k, const float *rot_v, const float *boundaries,
                const uint16_t *k, const uint16_t *v, const int32_t *slots, int n,
                uint8_t *pages, double *margin_k, double *margin_v) {
  size_t vb = rqo_vector_bytes(bits, d);
  size_t pb = rqo_page_bytes(bits, page_size, d);
  uint8_t codes[1024];
  for (int t = 0; t < n; ++t) {
    int s = slots[t];
    if (s < 0) continue;
    int page = s / page_size, off = s % page_size;
    for (int h = 0; h < hkv; ++h) {
      uint8_t *chunk = pages + ((size_t)page * hkv + h) * pb;
      const size_t src = ((size_t)t * hkv + h) * d;
      uint16_t nk, nv;
      rqo_encode(mode, bits, d, rot_k + (size_t)h * rot_stride(mode, d), boundaries, k + src, codes, &nk,
                 margin_k ? margin_k + src : NULL);
      rqo_pack(bits, d, codes, chunk + off * vb);
      rqo_encode(mode, bits, d, rot_v + (size_t)h * rot_stride(mode, d), boundaries, v + src, codes, &nv,
                 margin_v ? margin_v + src : NULL);
      uint8_t packed[1024];
      rqo_pack(bits, d, codes, packed);
      put_v(bits, d, chunk + page_size * vb, off, packed);
      uint8_t *norms = chunk + 2 * page_size * vb;
      norms[2 * off] = (uint8_t)(nk & 0xff);
      norms[2 * off + 1] = (uint8_t)(nk >> 8);
      norms[2 * page_size + 2 * off] = (uint8_t)(nv & 0xff);
      norms[2 * page_size + 2 * off + 1] = (uint8_t)(nv >> 8);
    }
  }
}

/* Dequantise token `pos` of sequence row `bt` for kv head h from the paged cache. */
static void load_token(int mode, int bits, int d, int hkv, int page_size, const float *rot_k,
                       const float *rot_v, const float *centroids, const uint8_t *pages,
                       const int32_t *bt, int pos, int h, double *kh, double *vh) {
  size_t vb = rqo_vector_bytes(bits, d);
  size_t pb = rqo_page_bytes(bits, page_size, d);
  int page = bt[pos / page_size], off = pos % page_size;
  const uint8_t *chunk = pages + ((size_t)page * hkv + h) * pb;
  const uint8_t *norms = chunk + 2 * page_size * vb;
  uint16_t nk = (uint16_t)(norms[2 * off] | (norms[2 * off + 1] << 8));
  uint16_t nv = (uint16_t)(norms[2 * page_size + 2 * off] | (norms[2 * page_size + 2 * off + 1] << 8));
  uint8_t codes[1024];
  rqo_unpack(bits, d, chunk + off * vb, codes);
  rqo_dequant(mode, bits, d, rot_k + (size_t)h * rot_stride(mode, d), centroids, codes, nk, kh);
  uint8_t packed[1024];
  get_v(bits, d, chunk + page_size * vb, off, packed);
  rqo_unpack(bits, d, packed, codes);
  rqo_dequant(mode, bits, d, rot_v + (size_t)h * rot_stride(mode, d), centroids, codes, nv, vh);
}

/*
 * Attention over the dequantised cache, in the original (unrotated) space.
 *   q: fp16 [B][T][Hq][d];  out: double [B][T][Hq][d].
 *   Query head hq reads kv head hq / (Hq / Hkv).  seq_lens[b] counts every cached token,
 *   the T query tokens included (they are the last T positions, the drafts).
 *   Visibility of position t to query row j:
 *     chain (tree_mask NULL): t <= len - T + j;
 *     tree: t < len - T (the prefix), or draft i = t - (len - T) with bit i of tree_mask[b][j].
 *   s_t = sm_scale * <q, k_t>,  o = sum over visible t of softmax(s)_t v_t.  A row that sees no
 *   position, or a sequence with len = 0, gives zeros.
 */
static int attention_impl(int mode, int bits, int d, int hq, int hkv, int page_size,
                          const float *rot_k, const float *rot_v, const float *centroids, double sm_scale,
                          const uint16_t *q, int T, const uint64_t *tree_mask, const uint8_t *pages,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B, double *out) {
  int group = hq / hkv;
  for (int b = 0; b < B; ++b) {
    int len = seq_lens[b];
    const int32_t *bt = block_table + (size_t)b * max_pages;
    for (int h = 0; h < hkv; ++h) {
      double *K = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1) * d);
      double *V = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1) * d);
      double *s = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
      char *vis = (char *)malloc((size_t)(len > 0 ? len : 1));
      if (!K || !V || !s || !vis) { free(K); free(V); free(s); free(vis); return -1; }
      for (int t = 0; t < len; ++t)
        load_token(mode, bits, d, hkv, page_size, rot_k, rot_v, centroids, pages, bt, t, h,
                   K + (size_t)t * d, V + (size_t)t * d);
      for (int j = 0; j < T; ++j) {
        int any = 0;
        for (int t = 0; t < len; ++t) {
          if (!tree_mask) {
            vis[t] = t <= len - T + j;
          } else {
            int i = t - (len - T);
            vis[t] = i < 0 ? 1 : (int)((tree_mask[(size_t)b * T + j] >> i) & 1u);
          }
          any |= vis[t];
        }
        for (int g = 0; g < group; ++g) {
          int head = h * group + g;
          const uint16_t *qv = q + (((size_t)b * T + j) * hq + head) * d;
          double *o = out + (((size_t)b * T + j) * hq + head) * d;
          for (int i = 0; i < d; ++i) o[i] = 0.0;
          if (len <= 0 || !any) continue;
          double qd[1024];
          for (int i = 0; i < d; ++i) qd[i] = rqo_half_to_double(qv[i]);
          double mx = -INFINITY;
          for (int t = 0; t < len; ++t) {
            if (!vis[t]) continue;
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qd[i] * K[(size_t)t * d + i];
            s[t] = sm_scale * acc;
            if (s[t] > mx) mx = s[t];
          }
          double denom = 0.0;
          for (int t = 0; t < len; ++t) {
            if (!vis[t]) continue;
            s[t] = exp(s[t] - mx);
            denom += s[t];
          }
          for (int t = 0; t < len; ++t) {
            if (!vis[t]) continue;
            double p = s[t] / denom;
            for (int i = 0; i < d; ++i) o[i] += p * V[(size_t)t * d + i];
          }
        }
      }
      free(K); free(V); free(s); free(vis);
    }
  }
  return 0;
}

int rqo_attention(int mode, int bits, int d, int hq, int hkv, int page_size,
                  const float *rot_k, const float *rot_v, const float *centroids, double sm_scale,
                  const uint16_t *q, int T, const uint8_t *pages, const int32_t *block_table,
                  int max_pages, const int32_t *seq_lens, int B, double *out) {
  return attention_impl(mode, bits, d, hq, hkv, page_size, rot_k, rot_v, centroids, sm_scale, q, T, NULL, pages,
                        block_table, max_pages, seq_lens, B, out);
}

/* Tree verify: tree_mask uint64 [B][T], bit i of row j = query j sees draft i (T <= 64). */
int rqo_tree_attention(int mode, int bits, int d, int hq, int hkv, int page_size,
                       const float *rot_k, const float *rot_v, const float *centroids, double sm_scale,
                       const uint16_t *q, int T, const uint64_t *tree_mask, const uint8_t *pages,
                       const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B, double *out) {
  if (T < 1 || T > 64 || !tree_mask) return -2;
  return attention_impl(mode, bits, d, hq, hkv, page_size, rot_k, rot_v, centroids, sm_scale, q, T, tree_mask,
                        pages, block_table, max_pages, seq_lens, B, out);
}

/* Plain attention over unquantised fp16 K/V given densely as [B][L][Hkv][d] (the fidelity
   reference: the same definition with no codec in between). */
int rqo_attention_dense(int d, int hq, int hkv, double sm_scale, const uint16_t *q, int T,
                        const uint16_t *k, const uint16_t *v, int L, const int32_t *seq_lens,
                        int B, double *out) {
  int group = hq / hkv;
  double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!s) return -1;
  for (int b = 0; b < B; ++b) {
    int len = seq_lens[b];
    for (int j = 0; j < T; ++j) {
      int last = len - T + j;
      for (int head = 0; head < hq; ++head) {
        int h = head / group;
        const uint16_t *qv = q + (((size_t)b * T + j) * hq + head) * d;
        double *o = out + (((size_t)b * T + j) * hq + head) * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (len <= 0 || last < 0) continue;
        double mx = -INFINITY;
        for (int t = 0; t <= last; ++t) {
          const uint16_t *kv = k + (((size_t)b * L + t) * hkv + h) * d;
          double acc = 0.0;
          for (int i = 0; i < d; ++i) acc += rqo_half_to_double(qv[i]) * rqo_half_to_double(kv[i]);
          s[t] = sm_scale * acc;
          if (s[t] > mx) mx = s[t];
        }
        double denom = 0.0;
        for (int t = 0; t <= last; ++t) { s[t] = exp(s[t] - mx); denom += s[t]; }
        for (int t = 0; t <= last; ++t) {
          const uint16_t *vv = v + (((size_t)b * L + t) * hkv + h) * d;
          double p = s[t] / denom;
          for (int i = 0; i < d; ++i) o[i] += p * rqo_half_to_double(vv[i]);
        }
      }
    }
  }
  free(s);
  return 0;
}
