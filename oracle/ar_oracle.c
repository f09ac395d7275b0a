/*
 * ar_oracle.c -- plain, slow CPU oracle of the emulated sum all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file.  The CUDA library never includes, links
 * or calls it, and it shares no header, helper or table with that library.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * Every float addition below is therefore one IEEE-754 binary32 addition,
 * round-to-nearest-even, with no contraction and no reassociation.
 *
 * The pages this follows:
 *  [CAR]  "SGLang JIT custom all-reduce" notes (obnotes, Inference/sglang/
 *         jit_kernel/0-custom-all-reduce), §1 "一次处理多大一块" (16-byte
 *         vectors), §4 "求和 (reduce_impl)" (fp32 accumulator that starts at
 *         zero, ranks added in GPU order 0..M-1, one round-to-nearest
 *         conversion at the end), §5 "写回".
 *  [MGPU] handbook chapter "多 GPU 与 NCCL", §集合通信 (all-reduce: every
 *         rank gets the sum; all-reduce = reduce-scatter + all-gather) and
 *         §ring all-reduce (p ranks in a ring, data cut into p chunks, p-1
 *         reduce-scatter steps in which each rank sends one chunk to the next
 *         rank, which adds its own chunk, then p-1 all-gather steps).
 *  [NCCL] handbook chapter "集合通信：NCCL 的算法、协议与推理框架的定制
 *         all-reduce", §协议 table (LL: 4 B data + 4 B flag in every 8 B;
 *         LL128: 120 B data + 8 B flag in every 128 B; the receiver polls the
 *         flag).
 *
 * Readings where the pages leave a step open (each one is listed with its
 * reason in the design notes):
 *  - payload types: fp32, bf16, fp16; fp16 is treated exactly like bf16.
 *  - two-shot and ring chunk: C = ceil(N/n) rounded up to a whole 16-byte
 *    vector; chunk r = elements [rC, min((r+1)C, N)), possibly short or empty.
 *  - ring: chunk c is sent by rank c first, so it is summed in the order
 *    c, c+1, ..., c+n-1 (mod n); partial sums stay fp32 across hops and are
 *    rounded once, by the rank that completes the chunk.  The first hop adds
 *    two raw values (no zero start), so only the rank-order sum maps an
 *    all-(-0) input to +0.
 *  - LL line: u32 data word at byte 0, u32 flag at byte 4 (little-endian).
 *  - LL128 line: 30 fp32 payload words at bytes 0..119 (zero padding after the
 *    last element), u64 flag at bytes 120..127.
 *  - a line whose flag is not the expected step is not consumed: its
 *    destination is left untouched and it is counted as bad.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

static uint32_t bits_of(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float float_of(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* ------------------------------------------------------------------------ */
/* Payload conversions, written from the IEEE-754 definitions.              */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of a binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return float_of((uint32_t)h << 16); }

/* binary32 -> bf16, round to nearest, ties to even, on the 16 bits dropped.
 * A carry out of the significand moves into the exponent, which also turns
 * values past the largest bf16 into infinity.  NaN stays NaN (quiet bit). */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = bits_of(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t drop = u & 0xffffu;
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

/* binary16 -> binary32: sign, 5-bit exponent (bias 15), 10-bit fraction. */
float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t e = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t m = (uint32_t)h & 0x3ffu;
    float v;
    if (e == 0x1fu) {
        v = m ? float_of(0x7fc00000u | (m << 13)) : INFINITY;
    } else if (e == 0) {
        v = ldexpf((float)m, -24);               /* subnormal: m * 2^-24 */
    } else {
        v = ldexpf((float)(1024u + m), (int)e - 25); /* (1.m) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even, with binary16
 * subnormals and overflow to infinity. */
uint16_t orc_f32_to_f16(float x)
{
    uint32_t u = bits_of(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)                                   /* NaN */
        return (uint16_t)(sign | 0x7e00u | ((a >> 13) & 0x3ffu));
    if (a == 0x7f800000u)                                  /* infinity */
        return (uint16_t)(sign | 0x7c00u);
    int eb = (int)(a >> 23);                               /* biased exponent */
    if (eb == 0)               /* binary32 subnormal: < 2^-126, rounds to 0 */
        return sign;
    int E = eb - 127;                                      /* unbiased */
    if (E >= 16)                                           /* >= 65536 */
        return (uint16_t)(sign | 0x7c00u);
    uint32_t m = (a & 0x7fffffu) | 0x800000u;    /* value = m * 2^(eb-150) */
    /* exponent of one binary16 unit in the last place at this magnitude */
    int q = (E >= -14) ? E - 10 : -24;
    int shift = q - (eb - 150);                  /* >= 13 */
    if (shift > 25)                              /* value < quantum / 4 */
        return sign;
    uint32_t r = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (r & 1u)))
        r += 1u;
    uint32_t bits;
    if (E >= -14)        /* normal: r in [1024, 2048]; a carry bumps the exponent */
        bits = ((uint32_t)(E + 15) << 10) + (r - 1024u);
    else                 /* subnormal: r in [0, 1024]; 1024 is the smallest normal */
        bits = r;
    if (bits >= 0x7c00u)
        bits = 0x7c00u;
    return (uint16_t)(sign | bits);
}

void orc_bf16_to_f32_n(const uint16_t* h, float* f, size_t n)
{ for (size_t i = 0; i < n; ++i) f[i] = orc_bf16_to_f32(h[i]); }
void orc_f32_to_bf16_n(const float* f, uint16_t* h, size_t n)
{ for (size_t i = 0; i < n; ++i) h[i] = orc_f32_to_bf16(f[i]); }
void orc_f16_to_f32_n(const uint16_t* h, float* f, size_t n)
{ for (size_t i = 0; i < n; ++i) f[i] = orc_f16_to_f32(h[i]); }
void orc_f32_to_f16_n(const float* f, uint16_t* h, size_t n)
{ for (size_t i = 0; i < n; ++i) h[i] = orc_f32_to_f16(f[i]); }

/* ------------------------------------------------------------------------ */
/* Element access in the payload type.                                      */
/* ------------------------------------------------------------------------ */

static size_t elem_size(int dt) { return dt == ORC_F32 ? 4u : 2u; }

static float widen(const void* p, size_t i, int dt)
{
    if (dt == ORC_F32) return ((const float*)p)[i];
    uint16_t h = ((const uint16_t*)p)[i];
    return dt == ORC_BF16 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

static void narrow(void* p, size_t i, float v, int dt)
{
    if (dt == ORC_F32) ((float*)p)[i] = v;
    else if (dt == ORC_BF16) ((uint16_t*)p)[i] = orc_f32_to_bf16(v);
    else ((uint16_t*)p)[i] = orc_f32_to_f16(v);
}

/* ------------------------------------------------------------------------ */
/* One-shot: the all-reduce by its definition.                              */
/* ------------------------------------------------------------------------ */

/* out[r][i] = RN( (((+0 + x_0[i]) + x_1[i]) + ...) + x_{n-1}[i] ) for every
 * rank r, fp32 accumulation, ranks in order 0..n-1 ([CAR] §4).  Every rank
 * gets the same bits ([MGPU] §集合通信). */
void orc_all_reduce(int n, const void* const* in, void* const* out, size_t N, int dt)
{
    for (size_t i = 0; i < N; ++i) {
        float acc = 0.0f;
        for (int r = 0; r < n; ++r)
            acc = acc + widen(in[r], i, dt);
        for (int r = 0; r < n; ++r)
            narrow(out[r], i, acc, dt);
    }
}

/* ------------------------------------------------------------------------ */
/* Two-shot: reduce-scatter, then all-gather ([MGPU] §集合通信).            */
/* ------------------------------------------------------------------------ */

/* Elements per chunk: ceil(N/n) rounded up to a whole 16-byte vector. */
size_t orc_chunk_elems(int n, size_t N, int dt)
{
    size_t per = (N + (size_t)n - 1) / (size_t)n;
    size_t q = 16u / elem_size(dt);
    return (per + q - 1) / q * q;
}

static void chunk_range(int c, size_t C, size_t N, size_t* lo, size_t* hi)
{
    size_t a = (size_t)c * C, b = a + C;
    if (a > N) a = N;
    if (b > N) b = N;
    *lo = a;
    *hi = b;
}

/* Rank r ends with the sum of chunk r, in out[r], rank order as one-shot. */
void orc_reduce_scatter(int n, const void* const* in, void* const* out, size_t N, int dt)
{
    size_t C = orc_chunk_elems(n, N, dt), lo, hi;
    for (int r = 0; r < n; ++r) {
        chunk_range(r, C, N, &lo, &hi);
        for (size_t i = lo; i < hi; ++i) {
            float acc = 0.0f;
            for (int q = 0; q < n; ++q)
                acc = acc + widen(in[q], i, dt);
            narrow(out[r], i, acc, dt);
        }
    }
}

/* Every rank copies chunk j from rank j, for every j. */
void orc_all_gather(int n, void* const* out, size_t N, int dt)
{
    size_t C = orc_chunk_elems(n, N, dt), lo, hi, e = elem_size(dt);
    for (int j = 0; j < n; ++j) {
        chunk_range(j, C, N, &lo, &hi);
        for (int r = 0; r < n; ++r)
            if (r != j && hi > lo)
                memcpy((char*)out[r] + lo * e, (const char*)out[j] + lo * e, (hi - lo) * e);
    }
}

/* ------------------------------------------------------------------------ */
/* Ring: the 2(n-1) steps of [MGPU] §ring all-reduce, simulated literally.  */
/* ------------------------------------------------------------------------ */

/* The ring's all-gather phase, steps s = 0..n-2: every rank r passes the
 * completed chunk (r + 1 - s) mod n it holds to rank r + 1.  All sends of a
 * step are taken from the state before the step.  On entry rank r holds
 * chunk (r + 1) mod n complete in out[r]. */
int orc_all_gather_ring(int n, void* const* out, size_t N, int dt)
{
    size_t C = orc_chunk_elems(n, N, dt), lo, hi, e = elem_size(dt);
    char* snap = (char*)malloc(e * (size_t)n * (C ? C : 1));
    if (!snap) return -1;
    for (int s = 0; s < n - 1; ++s) {
        for (int r = 0; r < n; ++r) {
            int c = ((r + 1 - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            if (hi > lo)
                memcpy(snap + (size_t)r * C * e, (const char*)out[r] + lo * e, (hi - lo) * e);
        }
        for (int r = 0; r < n; ++r) {
            int d = (r + 1) % n, c = ((r + 1 - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            if (hi > lo)
                memcpy((char*)out[d] + lo * e, snap + (size_t)r * C * e, (hi - lo) * e);
        }
    }
    free(snap);
    return 0;
}

/* Each rank keeps an fp32 working copy of its buffer.  Reduce-scatter step
 * s = 0..n-2: every rank r sends its chunk c = (r - s) mod n to rank
 * d = (r + 1) mod n, which adds it to its own chunk c.  After n-1 steps rank
 * r holds the full sum of chunk (r + 1) mod n and rounds it once.
 * All-gather step s = 0..n-2: every rank r passes its completed chunk
 * (r + 1 - s) mod n to rank r + 1.  All sends of a step are taken from the
 * state before the step. */
int orc_ring(int n, const void* const* in, void* const* out, size_t N, int dt)
{
    size_t C = orc_chunk_elems(n, N, dt), lo, hi, e = elem_size(dt);
    float* work = (float*)malloc(sizeof(float) * (size_t)n * (N ? N : 1));
    float* sent = (float*)malloc(sizeof(float) * (size_t)n * (C ? C : 1));
    if (!work || !sent) { free(work); free(sent); return -1; }

    for (int r = 0; r < n; ++r)
        for (size_t i = 0; i < N; ++i)
            work[(size_t)r * N + i] = widen(in[r], i, dt);

    for (int s = 0; s < n - 1; ++s) {
        for (int r = 0; r < n; ++r) {                     /* everyone sends */
            int c = ((r - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            for (size_t i = lo; i < hi; ++i)
                sent[(size_t)r * C + (i - lo)] = work[(size_t)r * N + i];
        }
        for (int r = 0; r < n; ++r) {                     /* next rank adds */
            int d = (r + 1) % n, c = ((r - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            for (size_t i = lo; i < hi; ++i)
                work[(size_t)d * N + i] = sent[(size_t)r * C + (i - lo)] + work[(size_t)d * N + i];
        }
    }
    for (int r = 0; r < n; ++r) {                         /* one rounding */
        chunk_range((r + 1) % n, C, N, &lo, &hi);
        for (size_t i = lo; i < hi; ++i)
            narrow(out[r], i, work[(size_t)r * N + i], dt);
    }
    free(work);
    free(sent);
    orc_all_gather_ring(n, out, N, dt);
    return 0;
}

/* The order the ring produces, stated per element: element i of chunk c gets
 * RN( x_c + x_{c+1} + ... + x_{c+n-1} ) (indices mod n, left to right, fp32).
 * cols[r][k] is rank r's value of the k-th sampled element and chunk[k] its
 * chunk index; the result goes to res[k]. */
void orc_ring_order_sum(int n, const void* const* cols, const int32_t* chunk,
                        void* res, size_t M, int dt)
{
    for (size_t k = 0; k < M; ++k) {
        int c = chunk[k];
        float acc = widen(cols[c % n], k, dt);
        for (int j = 1; j < n; ++j)
            acc = acc + widen(cols[(c + j) % n], k, dt);
        narrow(res, k, acc, dt);
    }
}

/* ------------------------------------------------------------------------ */
/* LL and LL128 protocol lines ([NCCL] §协议).                              */
/* ------------------------------------------------------------------------ */

static void put_u32(uint8_t* p, uint32_t v)
{ p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24); }
static uint32_t get_u32(const uint8_t* p)
{ return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24); }
static void put_u64(uint8_t* p, uint64_t v) { put_u32(p, (uint32_t)v); put_u32(p + 4, (uint32_t)(v >> 32)); }
static uint64_t get_u64(const uint8_t* p) { return (uint64_t)get_u32(p) | ((uint64_t)get_u32(p + 4) << 32); }

/* LL: one 8-byte line per fp32 payload word. */
size_t orc_ll_bytes(size_t count) { return 8u * count; }

void orc_ll_pack(const float* src, uint8_t* lines, size_t count, uint32_t step)
{
    for (size_t i = 0; i < count; ++i) {
        put_u32(lines + 8 * i, bits_of(src[i]));
        put_u32(lines + 8 * i + 4, step);
    }
}

/* Returns the number of lines whose flag is not `step` (left unconsumed). */
size_t orc_ll_unpack(const uint8_t* lines, float* dst, size_t count, uint32_t step)
{
    size_t bad = 0;
    for (size_t i = 0; i < count; ++i) {
        if (get_u32(lines + 8 * i + 4) != step) { ++bad; continue; }
        dst[i] = float_of(get_u32(lines + 8 * i));
    }
    return bad;
}

/* Flag-checked reduce: a line is consumed only when every rank's copy of it
 * carries `step`; then its words are summed in rank order (fp32, from +0) and
 * written to every rank's output line with flag `step`. */
size_t orc_ll_reduce(int n, const uint8_t* const* in, uint8_t* const* out, size_t count, uint32_t step)
{
    size_t bad = 0;
    for (size_t i = 0; i < count; ++i) {
        int ok = 1;
        for (int r = 0; r < n; ++r)
            ok = ok && get_u32(in[r] + 8 * i + 4) == step;
        if (!ok) { ++bad; continue; }
        float acc = 0.0f;
        for (int r = 0; r < n; ++r)
            acc = acc + float_of(get_u32(in[r] + 8 * i));
        for (int r = 0; r < n; ++r) {
            put_u32(out[r] + 8 * i, bits_of(acc));
            put_u32(out[r] + 8 * i + 4, step);
        }
    }
    return bad;
}

/* LL128: 30 fp32 payload words and one u64 flag per 128-byte line. */
size_t orc_ll128_lines(size_t count) { return (count + 29u) / 30u; }
size_t orc_ll128_bytes(size_t count) { return 128u * orc_ll128_lines(count); }

void orc_ll128_pack(const float* src, uint8_t* lines, size_t count, uint64_t step)
{
    size_t L = orc_ll128_lines(count);
    for (size_t k = 0; k < L; ++k) {
        uint8_t* line = lines + 128 * k;
        for (size_t j = 0; j < 30; ++j) {
            size_t idx = 30 * k + j;
            put_u32(line + 4 * j, idx < count ? bits_of(src[idx]) : 0u);
        }
        put_u64(line + 120, step);
    }
}

size_t orc_ll128_unpack(const uint8_t* lines, float* dst, size_t count, uint64_t step)
{
    size_t L = orc_ll128_lines(count), bad = 0;
    for (size_t k = 0; k < L; ++k) {
        const uint8_t* line = lines + 128 * k;
        if (get_u64(line + 120) != step) { ++bad; continue; }
        for (size_t j = 0; j < 30; ++j) {
            size_t idx = 30 * k + j;
            if (idx < count) dst[idx] = float_of(get_u32(line + 4 * j));
        }
    }
    return bad;
}

/* All 30 words of a line are summed, padding included, so the output line's
 * padding is the sum of the inputs' padding (zero for packed inputs). */
size_t orc_ll128_reduce(int n, const uint8_t* const* in, uint8_t* const* out, size_t count, uint64_t step)
{
    size_t L = orc_ll128_lines(count), bad = 0;
    for (size_t k = 0; k < L; ++k) {
        int ok = 1;
        for (int r = 0; r < n; ++r)
            ok = ok && get_u64(in[r] + 128 * k + 120) == step;
        if (!ok) { ++bad; continue; }
        for (size_t j = 0; j < 30; ++j) {
            float acc = 0.0f;
            for (int r = 0; r < n; ++r)
                acc = acc + float_of(get_u32(in[r] + 128 * k + 4 * j));
            for (int r = 0; r < n; ++r)
                put_u32(out[r] + 128 * k + 4 * j, bits_of(acc));
        }
        for (int r = 0; r < n; ++r)
            put_u64(out[r] + 128 * k + 120, step);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* All-reduce fused with residual add and RMSNorm (the decode epilogue).     */
/* ------------------------------------------------------------------------ */

/* The handbook chapter "集合通信：NCCL 的算法、协议…" (§源码对照) names an
 * all-reduce + RMSNorm fused kernel for tensor-parallel layers without
 * defining it; the reading taken is that fusing changes nothing in the
 * result of the unfused chain:
 *   a[t][h]   = the all-reduce of in[*][t][h] (rank-order fp32 sum, rounded)
 *   r[t][h]   = RN( a + residual[t][h] )            -> residual_out
 *   y[t][h]   = RN( r * 1/sqrt(mean_h(r^2) + eps) * weight[h] ) -> norm_out
 * The mean of squares and the scaling are computed here in double (the
 * kernel's order of summation over h is its own); y is therefore compared
 * within one payload ulp, a and r bit for bit. */
void orc_allreduce_rmsnorm(int n, const void* const* in, const void* residual, const void* weight, double eps,
                           void* norm_out, void* residual_out, size_t T, size_t H, int dt)
{
    for (size_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (size_t h = 0; h < H; ++h) {
            size_t i = t * H + h;
            float acc = 0.0f;
            for (int r = 0; r < n; ++r)
                acc = acc + widen(in[r], i, dt);
            narrow(residual_out, i, acc, dt);                       /* a, rounded */
            float rr = widen(residual_out, i, dt) + widen(residual, i, dt);
            narrow(residual_out, i, rr, dt);                        /* r, rounded */
            double rv = (double)widen(residual_out, i, dt);
            ss += rv * rv;
        }
        double inv = 1.0 / sqrt(ss / (double)H + eps);
        for (size_t h = 0; h < H; ++h) {
            size_t i = t * H + h;
            double y = (double)widen(residual_out, i, dt) * inv * (double)widen(weight, h, dt);
            narrow(norm_out, i, (float)y, dt);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Ring with partials rounded to the payload type at every hop.             */
/* ------------------------------------------------------------------------ */

/* The same 2(n-1) steps as orc_ring, but what a rank sends on is its
 * partial sum rounded to the payload type, as a library that keeps its
 * buffers in the payload type does: chunk c gets
 *   RN( ... RN( RN(x_c + x_{c+1}) + x_{c+2} ) ... + x_{c+n-1} )
 * with each + one binary32 addition.  For fp32 payloads it equals orc_ring. */
int orc_ring_rounded(int n, const void* const* in, void* const* out, size_t N, int dt)
{
    size_t C = orc_chunk_elems(n, N, dt), lo, hi, e = elem_size(dt);
    char* work = (char*)malloc(e * (size_t)n * (N ? N : 1));  /* each rank's buffer, payload type */
    char* sent = (char*)malloc(e * (size_t)n * (C ? C : 1));
    if (!work || !sent) { free(work); free(sent); return -1; }
    for (int r = 0; r < n; ++r)
        memcpy(work + (size_t)r * N * e, in[r], N * e);
    for (int s = 0; s < n - 1; ++s) {
        for (int r = 0; r < n; ++r) {
            int c = ((r - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            if (hi > lo)
                memcpy(sent + (size_t)r * C * e, work + ((size_t)r * N + lo) * e, (hi - lo) * e);
        }
        for (int r = 0; r < n; ++r) {
            int d = (r + 1) % n, c = ((r - s) % n + n) % n;
            chunk_range(c, C, N, &lo, &hi);
            for (size_t i = lo; i < hi; ++i) {
                float v = widen(sent, (size_t)r * C + (i - lo), dt) + widen(work, (size_t)d * N + i, dt);
                narrow(work, (size_t)d * N + i, v, dt);
            }
        }
    }
    /* rank r holds chunk r+1 complete; the all-gather passes the chunks on */
    for (int r = 0; r < n; ++r) {
        chunk_range((r + 1) % n, C, N, &lo, &hi);
        if (hi > lo)
            memcpy((char*)out[r] + lo * e, work + ((size_t)r * N + lo) * e, (hi - lo) * e);
    }
    free(sent);
    free(work);
    orc_all_gather_ring(n, out, N, dt);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Pairwise (recursive-doubling) tree.                                      */
/* ------------------------------------------------------------------------ */

/* The PCIe-IPC blog post (bhfrc.com/news/61376, §3.1 算法骨架) pairs the
 * ranks up and, in each of log2(n) levels, lets each rank read its own and its peer's data, add, and
 * write the sum back to both.  Reading: at level l rank r pairs with
 * r XOR 2^l; the buffers hold the payload type, so each level's sum is one
 * binary32 add of the two widened values, rounded to the payload type.  n
 * must be a power of two.  Both members of a pair add the same two values
 * (a + b == b + a), so every rank ends with the same bits.  Returns -1 when
 * n is not a power of two. */
int orc_tree(int n, const void* const* in, void* const* out, size_t N, int dt)
{
    if (n < 2 || (n & (n - 1))) return -1;
    size_t e = elem_size(dt);
    char* cur = (char*)malloc(e * (size_t)n * (N ? N : 1));
    char* nxt = (char*)malloc(e * (size_t)n * (N ? N : 1));
    if (!cur || !nxt) { free(cur); free(nxt); return -2; }
    for (int r = 0; r < n; ++r)
        memcpy(cur + (size_t)r * N * e, in[r], N * e);
    for (int d = 1; d < n; d <<= 1) {
        for (int r = 0; r < n; ++r) {
            int p = r ^ d;
            for (size_t i = 0; i < N; ++i) {
                float v = widen(cur, (size_t)r * N + i, dt) + widen(cur, (size_t)p * N + i, dt);
                narrow(nxt, (size_t)r * N + i, v, dt);
            }
        }
        char* t = cur; cur = nxt; nxt = t;
    }
    for (int r = 0; r < n; ++r)
        memcpy(out[r], cur + (size_t)r * N * e, N * e);
    free(cur);
    free(nxt);
    return 0;
}
