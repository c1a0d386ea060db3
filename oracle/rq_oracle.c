/*
 * rq_oracle.c -- plain CPU oracle for the inverse-RoPE + block-FP8 quant
 * epilogue and its forward-RoPE + paged-insert sibling.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, scalar statement of what the
 * CUDA library must compute.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg load it.  It shares no code,
 * header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        -pthread rq_oracle.c -lm
 * (-ffp-contract=off keeps every product and sum separately rounded to
 * fp32, as the op order below states.)
 *
 * Sources, cited by page title and section:
 *  [INV] "[vllm] 한 프로그램이 4개 head를 처리하게 하라: DeepSeek-V4 inverse
 *        RoPE + FP8 quant 커널 3.5배 가속기" (analysis of vLLM PR #63540).
 *        Intro: bf16 [token, head, 512] input, inverse RoPE then block FP8.
 *        S1 (BLOCK_H): output group g = head // heads_per_group, position
 *        of the head inside its group, per-head scale slot = 4 * that.
 *        S2 (register swap): the GPT-J (even, odd) pair rotation of the
 *        last 64 dims, cos in cache columns 0..31, sin in 32..63.
 *        S3 (3-D quant): amax over 128-element blocks, clamped below by eps.
 *  [KV]  "[vllm] vLLM DeepSeek-V4 성능 최적화: Eager Break 시 Workspace 재사용
 *        개선" (analysis of vLLM PR #49236), S1: kv [N, 512] is rotated,
 *        quantised and inserted into a paged uint8 k_cache by slot_mapping.
 *  [IDX] "[vllm] vLLM의 GLM5.2 성능 최적화: Triton 커널 융합을 통한 E2E
 *        Throughput 향상" (analysis of vLLM PR #46862), S1: the power-of-two
 *        scale exp2(ceil(log2(raw scale))).
 *  [IDX] S1 also shows the indexer kernel's steps: RoPE output rounded
 *        through bf16, power-of-two FP8 scale, and the scale folded into the
 *        indexer weights as weight * q_scale * softmax_scale * head_scale.
 *  [OFP8] OCP 8-bit Floating Point Specification (OFP8) rev 1.0: E4M3
 *        (bias 7, no infinities, S.1111.111 is NaN, max normal 448).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes of the repository):
 *  - raw scale = fl32(amax / 448) (the FP8 maximum of E4M3); the exponent is
 *    the exact ceiling of log2 of that fp32 value;
 *  - e4m3 encode rounds to nearest, ties to even, and saturates finite and
 *    infinite magnitudes at 448; NaN encodes as 0x7F; zero keeps its sign;
 *  - rotation: two separately rounded fp32 products, then one rounded fp32
 *    add or subtract, in the order the page writes them;
 *  - the forward rotation (insert sibling) is the rotation by +theta, the
 *    inverse one by -theta;
 *  - paged record of one token: 512 code bytes then the 4 fp32 block scales
 *    (528 bytes) at k_cache + (slot / block_size) * block_stride
 *    + (slot % block_size) * 528; a negative slot means "skip this token".
 *  - UE8M0 scale packing ([INV] S3 mentions it without a layout): each
 *    power-of-two block scale 2^e becomes the byte e + 127 (the OCP
 *    Microscaling E8M0 encoding, value 2^(byte - 127)), and the four blocks
 *    of a head are packed into one 32-bit word, block b in bits 8b..8b+7;
 *  - the non-quantising variant ([INV] S4, CompileKey.quantize): the
 *    inverse-rotated head is written as bf16, each fp32 value rounded to
 *    the nearest bf16, ties to even, in the same [N, G, hpg*512] layout.
 *  - the fused q/kv op ([KV] S1): each q head (512 wide) is RMS-normalised
 *    over its 512 values, x / sqrt(mean(x^2) + eps), times an optional
 *    per-dimension weight (the page's op takes none: NULL; with one, the
 *    usual RMSNorm convention, the weight multiplies before the rotation),
 *    then forward-rotated like kv, and written as bf16 into a
 *    q_out padded to q_head_padded heads, the pad heads all zero; kv is the
 *    insert op above. The oracle computes the q part in double and rounds
 *    the double result straight to bf16 (the pages fix no precision for it).
 *  - the indexer q op ([IDX] S1): q heads are 128 wide, dims 0..63 rotated
 *    forward (NeoX halves: x0 = dim j, x1 = dim 32 + j; or GPT-J pairs:
 *    x0 = dim 2j, x1 = dim 2j + 1), r0 = x0*c - x1*s, r1 = x1*c + x0*s with
 *    every product and sum rounded to fp32, then rounded to bf16 and back;
 *    one block per head: amax over its 128 values clamped by eps, the same
 *    power-of-two scale, e4m3 codes; the scale is folded into the head's
 *    weight, ((weight * q_scale) * softmax_scale) * head_scale in fp32.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HEAD_DIM 512        /* [INV] intro: 512-wide heads            */
#define NOPE_DIM 448        /* [INV] S2: pairs >= NOPE_DIM/2 are RoPE  */
#define HALF_ROPE 32        /* [INV] S2: sin starts at column 32       */
#define QUANT_BLOCK 128     /* [INV] S3: QUANT_GROUP_SIZE              */
#define BLOCKS_PER_HEAD 4   /* [INV] S3: CHUNKS_PER_HEAD = 512 / 128   */
#define CACHE_WIDTH 64      /* [KV] S1: cos_sin_cache.size(1) == 64    */
#define RECORD_BYTES 528    /* paged record: 512 codes + 4 fp32 scales */
#define E4M3_MAX 448.0      /* [OFP8] largest finite E4M3 magnitude    */

/* status codes of the oracle's own argument checks */
#define RQO_OK 0
#define RQO_ERR_ARG 1
#define RQO_ERR_GROUPING 4
#define RQO_ERR_POSITION 6
#define RQO_ERR_SLOT 7

/* ---------------------------------------------------------------- scalars */

/* bf16 is the upper half of an IEEE-754 binary32 pattern, so widening is a
 * 16-bit shift and exact ([INV] S1: the tile is loaded and converted to fp32). */
float rqo_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* [OFP8] E4M3 decode: s eeee mmm; e == 0 is subnormal m/8 * 2^-6,
 * otherwise (1 + m/8) * 2^(e-7); s 1111 111 is NaN. */
/* Nearest bf16 to an fp32 value, ties to even (IEEE-754 round to nearest on
 * the 16 dropped bits; a carry out of the mantissa correctly moves to the
 * next binade or to infinity). NaN stays NaN (sign kept, quiet bit set). */
uint16_t rqo_f32_to_bf16(float f)
{
    uint32_t u, lo, hi;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    hi = u >> 16;
    lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u;
    return (uint16_t)hi;
}

/* Nearest bf16 to a double, ties to even, rounded once (no detour through
 * fp32): v = m * 2^E with 0.5 <= |m| < 1 keeps 8 significant bits (4 fewer
 * below the bf16 normal range, down to the smallest subnormal 2^-133).
 * Results beyond the largest finite bf16 become infinities. */
uint16_t rqo_f64_to_bf16(double v)
{
    double m, r;
    int E, keep;
    float f;
    uint32_t u;
    if (v != v)
        return 0x7fc0u;
    if (v == 0.0 || isinf(v)) {
        f = (float)v;               /* exact: zero or infinity keeps its sign */
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    m = frexp(v, &E);               /* v = m * 2^E, 0.5 <= |m| < 1 */
    keep = 8;                       /* bf16: 8 significant bits when normal */
    if (E - 1 < -126)               /* below 2^-126: subnormal spacing 2^-133 */
        keep = 8 - (-126 - (E - 1));
    if (keep < 0)
        return (uint16_t)(v < 0 ? 0x8000u : 0u);
    r = nearbyint(ldexp(m, keep));  /* default rounding mode: to nearest, ties to even */
    r = ldexp(r, E - keep);
    if (fabs(r) > 3.3895313892515355e38)  /* (2 - 2^-7) * 2^127, the largest bf16 */
        return (uint16_t)(v < 0 ? 0xff80u : 0x7f80u);
    f = (float)r;                   /* exact: r has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* OCP Microscaling E8M0 byte of a power-of-two scale 2^e (e in [-127, 127]):
 * e + 127. frexp gives s = 0.5 * 2^E exactly for a power of two, so e = E - 1. */
uint8_t rqo_ue8m0_of_scale(float s)
{
    int E;
    (void)frexp((double)s, &E);
    return (uint8_t)(E - 1 + 127);
}

/* Four block scales of a head packed as UE8M0 bytes, block b in bits 8b..8b+7. */
uint32_t rqo_pack_ue8m0(const float *scales4)
{
    uint32_t w = 0;
    int b;
    for (b = 0; b < BLOCKS_PER_HEAD; ++b)
        w |= (uint32_t)rqo_ue8m0_of_scale(scales4[b]) << (8 * b);
    return w;
}

double rqo_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    mag = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -mag : mag;
}

/* [OFP8] E4M3 encode of a real value v (given exactly as a double): round
 * to the nearest representable value, ties to an even mantissa; magnitudes
 * at or beyond 448 (and infinities) saturate to 448; NaN -> 0x7F. */
uint8_t rqo_e4m3_encode(double v)
{
    uint8_t sign;
    double a, quantum, r;
    int ex, e2;

    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs(v);
    if (a == 0.0)
        return sign;
    if (a >= E4M3_MAX)
        return sign | 0x7E;
    /* a = f * 2^ex2 with f in [0.5, 1): the binade of a is 2^(ex2-1). */
    frexp(a, &ex);
    ex -= 1;
    if (ex < -6)
        ex = -6;                      /* subnormal binade shares 2^-6's step */
    quantum = ldexp(1.0, ex - 3);     /* 3 mantissa bits -> 8 steps a binade */
    r = nearbyint(a / quantum) * quantum; /* a / quantum is exact (power of 2);
                                             nearbyint rounds ties to even */
    if (r == 0.0)
        return sign;
    if (r >= E4M3_MAX)
        return sign | 0x7E;
    frexp(r, &e2);
    e2 -= 1;
    if (e2 < -6)                      /* subnormal: m * 2^-9, m = 1..7 */
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    return sign | (uint8_t)((e2 + 7) << 3) |
           (uint8_t)((int)(r / ldexp(1.0, e2 - 3)) - 8);
}

/* Exact ceil(log2(r)) for finite r > 0.  frexp writes r = f * 2^E with f in
 * [0.5, 1) (subnormals included, after widening to double); r is a power of
 * two exactly when f == 0.5, and then log2 r = E - 1; otherwise
 * E - 1 < log2 r < E. */
int rqo_ceil_log2(float r)
{
    int E;
    double f = frexp((double)r, &E);
    return (f == 0.5) ? E - 1 : E;
}

/* Power-of-two block scale, [IDX] S1 and the [INV] quant step:
 * scale = 2^ceil(log2(amax / 448)), the division rounded once to fp32.
 * amax is the already-clamped block absmax (>= eps). */
float rqo_block_scale(float amax)
{
    float raw = amax / 448.0f;
    return ldexpf(1.0f, rqo_ceil_log2(raw));
}

/* ------------------------------------------------------------- row steps */

/* [INV] S2 rotation of one 512-wide fp32 row in place.  Pair j (0..31) is
 * (row[448+2j], row[449+2j]) with cos = cs_row[j], sin = cs_row[32+j].
 * inverse != 0:  even' = even*cos + odd*sin,  odd' = odd*cos - even*sin
 * inverse == 0:  even' = even*cos - odd*sin,  odd' = odd*cos + even*sin
 * Dims 0..447 pass through. */
void rqo_rope_row(float *row, const float *cs_row, int inverse)
{
    int j;
    for (j = 0; j < HALF_ROPE; ++j) {
        float even = row[NOPE_DIM + 2 * j];
        float odd = row[NOPE_DIM + 2 * j + 1];
        float c = cs_row[j];
        float s = cs_row[HALF_ROPE + j];
        float ec = even * c, os = odd * s, oc = odd * c, es = even * s;
        if (inverse) {
            row[NOPE_DIM + 2 * j] = ec + os;
            row[NOPE_DIM + 2 * j + 1] = oc - es;
        } else {
            row[NOPE_DIM + 2 * j] = ec - os;
            row[NOPE_DIM + 2 * j + 1] = oc + es;
        }
    }
}

/* [INV] S3 block quant of one 512-wide fp32 row: for each 128-element block,
 * amax = max(max |y|, eps), scale = 2^ceil(log2(fl32(amax/448))),
 * code = E4M3(y / scale).  y / scale is exact in double (scale is a power
 * of two), so the only rounding is the E4M3 one. */
void rqo_quant_row(const float *row, float eps, uint8_t *codes, float *scales)
{
    int b, k;
    for (b = 0; b < BLOCKS_PER_HEAD; ++b) {
        const float *y = row + b * QUANT_BLOCK;
        float amax = 0.0f, scale;
        for (k = 0; k < QUANT_BLOCK; ++k) {
            float m = fabsf(y[k]);
            if (m > amax)
                amax = m;
        }
        if (amax < eps)
            amax = eps;
        scale = rqo_block_scale(amax);
        scales[b] = scale;
        for (k = 0; k < QUANT_BLOCK; ++k)
            codes[b * QUANT_BLOCK + k] =
                rqo_e4m3_encode((double)y[k] / (double)scale);
    }
}

/* ------------------------------------------------------------ array forms */

void rqo_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_e4m3_encode((double)v[i]);
}

void rqo_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_e4m3_decode(c[i]);
}

void rqo_ceil_log2_array(const float *r, int64_t n, int32_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_ceil_log2(r[i]);
}

void rqo_block_scale_array(const float *amax, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_block_scale(amax[i]);
}

/* rows: [R, 512] fp32, rotated in place with cache row pos[r] */
void rqo_f32_to_bf16_array(const float *v, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_f32_to_bf16(v[i]);
}

void rqo_f64_to_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = rqo_f64_to_bf16(v[i]);
}

void rqo_pack_ue8m0_array(const float *scales, int64_t heads, uint32_t *out)
{
    int64_t i;
    for (i = 0; i < heads; ++i)
        out[i] = rqo_pack_ue8m0(scales + i * BLOCKS_PER_HEAD);
}

int rqo_rope_rows(float *rows, int64_t R, const int64_t *pos,
                  const float *cache, int64_t cache_rows, int inverse)
{
    int64_t r;
    for (r = 0; r < R; ++r) {
        if (pos[r] < 0 || pos[r] >= cache_rows)
            return RQO_ERR_POSITION;
        rqo_rope_row(rows + r * HEAD_DIM, cache + pos[r] * CACHE_WIDTH,
                     inverse);
    }
    return RQO_OK;
}

/* rows: [R, 512] fp32 -> codes [R, 512], scales [R, 4] */
void rqo_quant_rows(const float *rows, int64_t R, float eps, uint8_t *codes,
                    float *scales)
{
    int64_t r;
    for (r = 0; r < R; ++r)
        rqo_quant_row(rows + r * HEAD_DIM, eps, codes + r * HEAD_DIM,
                      scales + r * BLOCKS_PER_HEAD);
}

/* --------------------------------------------------------- inverse op */

struct inv_args {
    const uint16_t *x;
    int64_t n_heads, sx_t, sx_h;
    const int64_t *pos;
    const float *cache;
    int64_t hpg;
    float eps;
    uint8_t *out;
    float *scales;
    int64_t t0, t1;
};

static void *inv_worker(void *p)
{
    const struct inv_args *a = (const struct inv_args *)p;
    const int64_t H = a->n_heads, hpg = a->hpg, G = H / hpg;
    float row[HEAD_DIM];
    int64_t t, h;
    int k;
    for (t = a->t0; t < a->t1; ++t) {
        const float *cs_row = a->cache + a->pos[t] * CACHE_WIDTH;
        for (h = 0; h < H; ++h) {
            /* [INV] S1: group and place of the head in its group */
            int64_t g = h / hpg, hig = h % hpg;
            const uint16_t *src = a->x + t * a->sx_t + h * a->sx_h;
            /* out [N, G, hpg*512]: head hig of group g owns bytes
             * [hig*512, hig*512 + 512) of row (t, g) */
            uint8_t *dst = a->out + ((t * G + g) * hpg + hig) * HEAD_DIM;
            /* scales [N, G, hpg*4]: block b of that head is qb = hig*4 + b */
            float *sdst = a->scales + (t * G + g) * (hpg * BLOCKS_PER_HEAD) +
                          hig * BLOCKS_PER_HEAD;
            for (k = 0; k < HEAD_DIM; ++k)
                row[k] = rqo_bf16_to_f32(src[k]);
            rqo_rope_row(row, cs_row, 1);
            rqo_quant_row(row, a->eps, dst, sdst);
        }
    }
    return NULL;
}

static int split_run(void *(*fn)(void *), void *args, size_t arg_size,
                     int64_t n_tokens, int nthreads,
                     void (*set_range)(void *, int64_t, int64_t))
{
    pthread_t tid[256];
    int started[256];
    unsigned char *buf;
    int i;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads > n_tokens)
        nthreads = (int)(n_tokens > 0 ? n_tokens : 1);
    buf = (unsigned char *)malloc(arg_size * (size_t)nthreads);
    if (!buf)
        return RQO_ERR_ARG;
    /* contiguous token ranges; each token's arithmetic does not depend on
     * which thread runs it */
    for (i = 0; i < nthreads; ++i) {
        int64_t t0 = n_tokens * i / nthreads, t1 = n_tokens * (i + 1) / nthreads;
        void *slot = buf + arg_size * (size_t)i;
        memcpy(slot, args, arg_size);
        set_range(slot, t0, t1);
        started[i] = nthreads > 1 && pthread_create(&tid[i], NULL, fn, slot) == 0;
        if (!started[i])
            fn(slot);
    }
    for (i = 0; i < nthreads; ++i)
        if (started[i])
            pthread_join(tid[i], NULL);
    free(buf);
    return RQO_OK;
}

static void inv_set_range(void *p, int64_t t0, int64_t t1)
{
    ((struct inv_args *)p)->t0 = t0;
    ((struct inv_args *)p)->t1 = t1;
}

/* Inverse RoPE + block-FP8 quant over a [N, H, 512] bf16 tensor with token
 * and head strides in elements.  out: [N, H/hpg, hpg*512] E4M3 codes,
 * scales: [N, H/hpg, hpg*4] fp32, both contiguous.  Tokens are split across
 * nthreads threads (each token is computed exactly as with one thread). */
int rqo_inv_rope_fp8_quant(const uint16_t *x, int64_t n_tokens,
                           int64_t n_heads, int64_t sx_t, int64_t sx_h,
                           const int64_t *pos, const float *cache,
                           int64_t cache_rows, int64_t hpg, float eps,
                           uint8_t *out, float *scales, int nthreads)
{
    struct inv_args a;
    int64_t t;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1 || !(eps > 0.0f))
        return RQO_ERR_ARG;
    if (hpg < 1 || n_heads % hpg != 0)
        return RQO_ERR_GROUPING;
    if (n_tokens == 0)
        return RQO_OK;
    if (!x || !pos || !cache || !out || !scales)
        return RQO_ERR_ARG;
    for (t = 0; t < n_tokens; ++t)
        if (pos[t] < 0 || pos[t] >= cache_rows)
            return RQO_ERR_POSITION;
    a.x = x;
    a.n_heads = n_heads;
    a.sx_t = sx_t;
    a.sx_h = sx_h;
    a.pos = pos;
    a.cache = cache;
    a.hpg = hpg;
    a.eps = eps;
    a.out = out;
    a.scales = scales;
    a.t0 = 0;
    a.t1 = n_tokens;
    return split_run(inv_worker, &a, sizeof a, n_tokens, nthreads,
                     inv_set_range);
}

/* The non-quantising variant: inverse RoPE of x [N, H, 512] bf16, written
 * as bf16 into out [N, H/hpg, hpg*512] (contiguous; head hig of group g at
 * [hig*512, hig*512 + 512) of row (t, g)). Single-threaded. */
int rqo_inv_rope_bf16(const uint16_t *x, int64_t n_tokens, int64_t n_heads,
                      int64_t sx_t, int64_t sx_h, const int64_t *pos,
                      const float *cache, int64_t cache_rows, int64_t hpg,
                      uint16_t *out)
{
    float row[HEAD_DIM];
    int64_t t, h, G;
    int k;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1)
        return RQO_ERR_ARG;
    if (hpg < 1 || n_heads % hpg != 0)
        return RQO_ERR_GROUPING;
    if (n_tokens == 0)
        return RQO_OK;
    if (!x || !pos || !cache || !out)
        return RQO_ERR_ARG;
    G = n_heads / hpg;
    for (t = 0; t < n_tokens; ++t) {
        if (pos[t] < 0 || pos[t] >= cache_rows)
            return RQO_ERR_POSITION;
        for (h = 0; h < n_heads; ++h) {
            int64_t g = h / hpg, hig = h % hpg;
            const uint16_t *src = x + t * sx_t + h * sx_h;
            uint16_t *dst = out + ((t * G + g) * hpg + hig) * HEAD_DIM;
            for (k = 0; k < HEAD_DIM; ++k)
                row[k] = rqo_bf16_to_f32(src[k]);
            rqo_rope_row(row, cache + pos[t] * CACHE_WIDTH, 1);
            for (k = 0; k < HEAD_DIM; ++k)
                dst[k] = rqo_f32_to_bf16(row[k]);
        }
    }
    return RQO_OK;
}

/* ---------------------------------------------------------- insert op */

struct ins_args {
    const uint16_t *kv;
    int64_t skv;
    const int64_t *pos;
    const float *cache;
    const int64_t *slots;
    uint8_t *k_cache;
    int64_t block_size, block_stride;
    float eps;
    int64_t t0, t1;
};

static void *ins_worker(void *p)
{
    const struct ins_args *a = (const struct ins_args *)p;
    float row[HEAD_DIM];
    float sc[BLOCKS_PER_HEAD];
    int64_t t;
    int k;
    for (t = a->t0; t < a->t1; ++t) {
        int64_t slot = a->slots[t];
        uint8_t *rec;
        if (slot < 0)
            continue; /* negative slot: token not cached */
        rec = a->k_cache + (slot / a->block_size) * a->block_stride +
              (slot % a->block_size) * RECORD_BYTES;
        for (k = 0; k < HEAD_DIM; ++k)
            row[k] = rqo_bf16_to_f32(a->kv[t * a->skv + k]);
        rqo_rope_row(row, a->cache + a->pos[t] * CACHE_WIDTH, 0);
        rqo_quant_row(row, a->eps, rec, sc);
        memcpy(rec + HEAD_DIM, sc, sizeof sc);
    }
    return NULL;
}

static void ins_set_range(void *p, int64_t t0, int64_t t1)
{
    ((struct ins_args *)p)->t0 = t0;
    ((struct ins_args *)p)->t1 = t1;
}

/* Forward RoPE + block-FP8 quant of kv [N, 512] bf16 (token stride skv
 * elements), each token's 528-byte record written to its slot of the paged
 * k_cache [num_blocks, block_stride] bytes.  Slots must be distinct. */
int rqo_rope_fp8_quant_insert(const uint16_t *kv, int64_t n_tokens,
                              int64_t skv, const int64_t *pos,
                              const float *cache, int64_t cache_rows,
                              const int64_t *slots, uint8_t *k_cache,
                              int64_t num_blocks, int64_t block_size,
                              int64_t block_stride, float eps, int nthreads)
{
    struct ins_args a;
    int64_t t;
    if (n_tokens < 0 || cache_rows < 1 || num_blocks < 1 || block_size < 1 ||
        block_stride < block_size * RECORD_BYTES || !(eps > 0.0f))
        return RQO_ERR_ARG;
    if (n_tokens == 0)
        return RQO_OK;
    if (!kv || !pos || !cache || !slots || !k_cache)
        return RQO_ERR_ARG;
    for (t = 0; t < n_tokens; ++t) {
        if (pos[t] < 0 || pos[t] >= cache_rows)
            return RQO_ERR_POSITION;
        if (slots[t] >= num_blocks * block_size)
            return RQO_ERR_SLOT;
    }
    a.kv = kv;
    a.skv = skv;
    a.pos = pos;
    a.cache = cache;
    a.slots = slots;
    a.k_cache = k_cache;
    a.block_size = block_size;
    a.block_stride = block_stride;
    a.eps = eps;
    a.t0 = 0;
    a.t1 = n_tokens;
    return split_run(ins_worker, &a, sizeof a, n_tokens, nthreads,
                     ins_set_range);
}

/* ------------------------------------------------- fused q + kv op ([KV] S1) */

/* One q head: RMS norm over its 512 values (times weight[k] when weight is
 * not NULL), forward rotation of dims 448..511, rounded once to bf16. All in
 * double. */
void rqo_qnorm_rope_row(const uint16_t *src, const float *cs_row, double eps,
                        const uint16_t *weight, uint16_t *dst)
{
    double y[HEAD_DIM], ss = 0.0, r;
    int k, j;
    for (k = 0; k < HEAD_DIM; ++k) {
        y[k] = (double)rqo_bf16_to_f32(src[k]);
        ss += y[k] * y[k];
    }
    r = 1.0 / sqrt(ss / HEAD_DIM + eps);
    for (k = 0; k < HEAD_DIM; ++k) {
        y[k] *= r;
        if (weight)            /* the norm's per-dimension weight, before the rotation */
            y[k] *= (double)rqo_bf16_to_f32(weight[k]);
    }
    for (j = 0; j < HALF_ROPE; ++j) {
        const double c = cs_row[j], s = cs_row[HALF_ROPE + j];
        const double e = y[NOPE_DIM + 2 * j], o = y[NOPE_DIM + 2 * j + 1];
        y[NOPE_DIM + 2 * j] = e * c - o * s;        /* forward: rotation by +theta */
        y[NOPE_DIM + 2 * j + 1] = o * c + e * s;
    }
    for (k = 0; k < HEAD_DIM; ++k)
        dst[k] = rqo_f64_to_bf16(y[k]);
}

/* q [N, Hq, 512] bf16 (strides sq_t, sq_h) -> q_out [N, Hpad, 512] bf16
 * contiguous (heads Hq..Hpad-1 zero); kv [N, 512] -> paged k_cache as in
 * rqo_rope_fp8_quant_insert (quant_eps is its block-amax clamp). */
int rqo_qnorm_rope_kv_rope_quant_insert(const uint16_t *q, int64_t n_tokens, int64_t n_heads_q,
                                        int64_t sq_t, int64_t sq_h, const uint16_t *kv,
                                        int64_t skv, uint16_t *q_out, int64_t q_head_padded,
                                        uint8_t *k_cache, int64_t num_blocks, int64_t block_size,
                                        int64_t block_stride, const int64_t *slots,
                                        const int64_t *pos, const float *cache,
                                        int64_t cache_rows, double norm_eps,
                                        const uint16_t *norm_weight, float quant_eps)
{
    int64_t t, h;
    int rc;
    if (n_tokens < 0 || n_heads_q < 1 || q_head_padded < n_heads_q || !(norm_eps >= 0.0))
        return RQO_ERR_ARG;
    if (n_tokens == 0)
        return RQO_OK;
    if (!q || !q_out)
        return RQO_ERR_ARG;
    for (t = 0; t < n_tokens; ++t) {
        if (pos[t] < 0 || pos[t] >= cache_rows)
            return RQO_ERR_POSITION;
        for (h = 0; h < q_head_padded; ++h) {
            uint16_t *dst = q_out + (t * q_head_padded + h) * HEAD_DIM;
            if (h < n_heads_q)
                rqo_qnorm_rope_row(q + t * sq_t + h * sq_h, cache + pos[t] * CACHE_WIDTH,
                                   norm_eps, norm_weight, dst);
            else
                memset(dst, 0, HEAD_DIM * sizeof *dst);
        }
    }
    rc = rqo_rope_fp8_quant_insert(kv, n_tokens, skv, pos, cache, cache_rows, slots, k_cache,
                                   num_blocks, block_size, block_stride, quant_eps, 1);
    return rc;
}

/* ---------------------------------------------- indexer q op ([IDX] S1) */

#define IDX_HEAD_DIM 128
#define IDX_ROPE_DIM 64

/* q [N, H, 128] bf16 (strides sq_t, sq_h) -> codes [N, H, 128] e4m3 and
 * weights_out [N, H] fp32 (weights [N, H] fp32 in). neox: 1 for NeoX halves,
 * 0 for GPT-J pairs. */
int rqo_indexer_q_rope_quant(const uint16_t *q, int64_t n_tokens, int64_t n_heads,
                             int64_t sq_t, int64_t sq_h, const int64_t *pos, const float *cache,
                             int64_t cache_rows, int neox, const float *weights,
                             float softmax_scale, float head_scale, float eps, uint8_t *codes,
                             float *weights_out)
{
    float y[IDX_HEAD_DIM];
    int64_t t, h;
    int k, j;
    if (n_tokens < 0 || n_heads < 1 || cache_rows < 1 || !(eps > 0.0f))
        return RQO_ERR_ARG;
    if (n_tokens == 0)
        return RQO_OK;
    if (!q || !pos || !cache || !weights || !codes || !weights_out)
        return RQO_ERR_ARG;
    for (t = 0; t < n_tokens; ++t) {
        const float *cs;
        if (pos[t] < 0 || pos[t] >= cache_rows)
            return RQO_ERR_POSITION;
        cs = cache + pos[t] * CACHE_WIDTH;
        for (h = 0; h < n_heads; ++h) {
            const uint16_t *src = q + t * sq_t + h * sq_h;
            float amax = 0.0f, scale, inv;
            for (k = 0; k < IDX_HEAD_DIM; ++k)
                y[k] = rqo_bf16_to_f32(src[k]);
            for (j = 0; j < IDX_ROPE_DIM / 2; ++j) {
                const int i0 = neox ? j : 2 * j, i1 = neox ? IDX_ROPE_DIM / 2 + j : 2 * j + 1;
                const float c = cs[j], s = cs[HALF_ROPE + j];
                const float x0 = y[i0], x1 = y[i1];
                const float a0 = x0 * c, b0 = x1 * s, a1 = x1 * c, b1 = x0 * s;
                const float r0 = a0 - b0, r1 = a1 + b1;
                y[i0] = rqo_bf16_to_f32(rqo_f32_to_bf16(r0));   /* .to(bf16).to(fp32) */
                y[i1] = rqo_bf16_to_f32(rqo_f32_to_bf16(r1));
            }
            for (k = 0; k < IDX_HEAD_DIM; ++k)
                if (fabsf(y[k]) > amax)
                    amax = fabsf(y[k]);
            if (amax < eps)
                amax = eps;
            scale = rqo_block_scale(amax);
            inv = 1.0f / scale;                        /* exact: a power of two */
            for (k = 0; k < IDX_HEAD_DIM; ++k)
                codes[(t * n_heads + h) * IDX_HEAD_DIM + k] = rqo_e4m3_encode((double)(y[k] * inv));
            {
                const float w0 = weights[t * n_heads + h] * scale;
                const float w1 = w0 * softmax_scale;
                weights_out[t * n_heads + h] = w1 * head_scale;
            }
        }
    }
    return RQO_OK;
}

/* ------------------------------------------------ bit-pattern range drivers */

/* Test drivers that apply the scalar steps above to every fp32 bit pattern of
 * a range [first, first + count) (count <= 2^32 - first), split over threads.
 * They add no arithmetic: each element is exactly what rqo_quant_row does to
 * one value or one block. */
struct range_args {
    uint32_t first;
    float eps;
    int e;
    float *scales;
    uint8_t *codes;
    int64_t t0, t1;
};

static float bits_to_f32(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static void range_set(void *p, int64_t t0, int64_t t1)
{
    ((struct range_args *)p)->t0 = t0;
    ((struct range_args *)p)->t1 = t1;
}

static void *block_scale_worker(void *p)
{
    const struct range_args *a = (const struct range_args *)p;
    int64_t i;
    for (i = a->t0; i < a->t1; ++i) {
        float amax = bits_to_f32(a->first + (uint32_t)i);
        if (amax < a->eps)
            amax = a->eps;            /* the clamp of rqo_quant_row */
        a->scales[i] = rqo_block_scale(amax);
    }
    return NULL;
}

static void *encode_worker(void *p)
{
    const struct range_args *a = (const struct range_args *)p;
    const double scale = ldexp(1.0, a->e);
    int64_t i;
    for (i = a->t0; i < a->t1; ++i)   /* the code step of rqo_quant_row */
        a->codes[i] = rqo_e4m3_encode((double)bits_to_f32(a->first + (uint32_t)i) / scale);
    return NULL;
}

/* scales[i] = block scale of a block whose absmax is the pattern first + i
 * (finite, >= 0), after the eps clamp. */
int rqo_block_scale_bits_range(uint32_t first, int64_t count, float eps, float *scales,
                               int nthreads)
{
    struct range_args a;
    if (count < 0 || (uint64_t)first + (uint64_t)count > ((uint64_t)1 << 32))
        return RQO_ERR_ARG;
    memset(&a, 0, sizeof a);
    a.first = first;
    a.eps = eps;
    a.scales = scales;
    return split_run(block_scale_worker, &a, sizeof a, count, nthreads, range_set);
}

/* codes[i] = E4M3 code of the pattern first + i divided by 2^e. */
int rqo_e4m3_encode_bits_range(uint32_t first, int64_t count, int e, uint8_t *codes,
                               int nthreads)
{
    struct range_args a;
    if (count < 0 || (uint64_t)first + (uint64_t)count > ((uint64_t)1 << 32))
        return RQO_ERR_ARG;
    memset(&a, 0, sizeof a);
    a.first = first;
    a.e = e;
    a.codes = codes;
    return split_run(encode_worker, &a, sizeof a, count, nthreads, range_set);
}
