/*
 * CPU oracle for the reduce and gather data movement of a custom collective.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. The CUDA
 * library never includes, links or calls it, and this file includes nothing
 * from the CUDA side: the two share no code.
 *
 * Every function below is the plain definition of what the collective
 * computes, written as scalar loops with no blocking, fusion or reordering:
 *
 *  - allreduce (one-shot and two-shot reach the same result): every rank's
 *    output is the element-wise sum of the W rank buffers.  Sources:
 *    "Question and suggestions about custom allreduce" (sglang discussion
 *    2918), the trt_reduce_internal.cu block comment quoted in yizhang2077's
 *    reply (each block pulls the chunk from every GPU and sums it into
 *    local_output), and leizhao1234's opening post (two-shot = reduce-scatter
 *    plus allgather of the reduced chunks).  The pages do not fix the
 *    accumulator; the reading taken here is an fp32 accumulator that starts
 *    from rank 0's value and adds ranks 1..W-1 in that order, then one
 *    round-to-nearest-even conversion to the element type.  int32 sums wrap
 *    modulo 2^32.
 *
 *  - allgather_into_tensor, rank-major: out[r*N + i] = in[r][i].  Source:
 *    "ccl: hierarchical cross-node AllGather (intra-node SDMA + inter-node
 *    RDMA) #441", the PR description (all_gather_into_tensor-compatible,
 *    bit-exact for bf16/fp16/fp32/int32).
 *
 *  - param-contiguous allgather (FSDP [param][rank] output): rank r's shard
 *    of param s lands at O_s*W + r*E_s, with O_s the sum of E_t for t < s.
 *    Source: the same PR, the commit that adds enqueue_param_contiguous.
 *
 * The element conversions are written from the IEEE 754 binary16 / binary32
 * definitions and the bfloat16 definition (the upper 16 bits of a binary32).
 * Build with -ffp-contract=off and without -ffast-math so that every float
 * addition is one IEEE binary32 addition.
 *
 * The *_mt entry points run the same loops with the element (or byte) index
 * range split over host threads (OpenMP, when the compiler offers it).  Each
 * output element is still computed by one thread with the same additions in
 * the same order, so their outputs are bit-identical to the single-threaded
 * ones; they exist only so that the CPU baseline can use every host core.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes used by this oracle's entry points */
enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1, ORACLE_FP32 = 2, ORACLE_INT32 = 3 };

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bfloat16 -> binary32: a bfloat16 is the top half of a binary32 word. */
float oracle_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even.
 * The 16 low fraction bits are dropped; the kept part is bumped by one unit
 * when the dropped part is above half a unit, or exactly half with the kept
 * part odd.  A carry out of the fraction raises the exponent, and a carry
 * past the largest finite value gives the infinity encoding, as IEEE wants.
 * NaN maps to a quiet NaN that keeps the sign and the leading payload bits. */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u = f32_to_bits(x);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
    return (uint16_t)kept;
}

/* binary16 -> binary32.  Fields: 1 sign, 5 exponent (bias 15), 10 fraction.
 * exponent 0 is zero or subnormal (m * 2^-24); exponent 31 is inf or NaN;
 * otherwise (1024 + m) * 2^(e - 25).  Both products are exact in binary32. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    float mag;
    if (e == 0) mag = ldexpf((float)m, -24);
    else if (e == 31) mag = m ? NAN : INFINITY;
    else mag = ldexpf((float)(m + 1024), e - 25);
    return sign ? -mag : mag;
}

/* binary32 -> binary16, round to nearest, ties to even.
 * The result is q * 2^E with an integer q: in the subnormal range
 * (|x| < 2^-14) the quantum is 2^-24; otherwise the quantum is 2^(k-10) where
 * 2^k <= |x| < 2^(k+1), so that q has 11 significant bits.  |x| / quantum is
 * exact in binary32 (scaling by a power of two); its integer part and
 * fraction are split exactly and rounded half-to-even.  Magnitudes from
 * 65520 (halfway between the largest finite half, 65504, and 2^16) up
 * round to infinity. */
uint16_t oracle_f32_to_f16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    float a = fabsf(x);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00u);
    int E;
    if (a < 0x1p-14f) {
        E = -24;
    } else {
        int ex;
        (void)frexpf(a, &ex);          /* a = f * 2^ex, 0.5 <= f < 1 */
        E = (ex - 1) - 10;
    }
    float n = ldexpf(a, -E);
    float whole = floorf(n);
    float frac = n - whole;
    uint32_t q = (uint32_t)whole;
    if (frac > 0.5f || (frac == 0.5f && (q & 1u))) q += 1u;
    if (E == -24) return (uint16_t)(sign | q);   /* q == 1024 encodes 2^-14 */
    int biased = E + 10 + 15;
    if (q == 2048u) { q = 1024u; biased += 1; }
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)(q - 1024u));
}

static float load_as_f32(const void *p, int dtype, int64_t i)
{
    switch (dtype) {
    case ORACLE_BF16: return oracle_bf16_to_f32(((const uint16_t *)p)[i]);
    case ORACLE_FP16: return oracle_f16_to_f32(((const uint16_t *)p)[i]);
    default:          return ((const float *)p)[i];
    }
}

static void store_from_f32(void *p, int dtype, int64_t i, float v)
{
    switch (dtype) {
    case ORACLE_BF16: ((uint16_t *)p)[i] = oracle_f32_to_bf16(v); break;
    case ORACLE_FP16: ((uint16_t *)p)[i] = oracle_f32_to_f16(v); break;
    default:          ((float *)p)[i] = v; break;
    }
}

static int elem_size(int dtype)
{
    switch (dtype) {
    case ORACLE_BF16: case ORACLE_FP16: return 2;
    case ORACLE_FP32: case ORACLE_INT32: return 4;
    default: return 0;
    }
}

/* Element-wise conversion between binary32 and one 16-bit format, for the
 * pins: exactly one of src_dtype / dst_dtype is ORACLE_FP32. */
int oracle_cast(const void *src, int src_dtype, void *dst, int dst_dtype, int64_t n)
{
    if (n < 0 || (n && (!src || !dst))) return -1;
    if (src_dtype == ORACLE_FP32 && (dst_dtype == ORACLE_BF16 || dst_dtype == ORACLE_FP16)) {
        for (int64_t i = 0; i < n; ++i) store_from_f32(dst, dst_dtype, i, ((const float *)src)[i]);
        return 0;
    }
    if (dst_dtype == ORACLE_FP32 && (src_dtype == ORACLE_BF16 || src_dtype == ORACLE_FP16)) {
        for (int64_t i = 0; i < n; ++i) ((float *)dst)[i] = load_as_f32(src, src_dtype, i);
        return 0;
    }
    return -1;
}

/* Allreduce: out[i] = sum over r = 0..W-1 of in[r][i].
 * Floating types: acc starts as in[0][i] widened to binary32, then
 * acc = acc + in[r][i] for r = 1, 2, ..., W-1, then one conversion.
 * int32: the same order, two's-complement wrap-around. */
int oracle_allreduce(const void *const *in, int W, int64_t numel, int dtype, void *out)
{
    if (W < 1 || numel < 0 || !in || elem_size(dtype) == 0) return -1;
    if (numel == 0) return 0;
    if (!out) return -1;
    for (int r = 0; r < W; ++r)
        if (!in[r]) return -1;
    if (dtype == ORACLE_INT32) {
        for (int64_t i = 0; i < numel; ++i) {
            uint32_t acc = (uint32_t)((const int32_t *)in[0])[i];
            for (int r = 1; r < W; ++r) acc += (uint32_t)((const int32_t *)in[r])[i];
            ((uint32_t *)out)[i] = acc;
        }
        return 0;
    }
    for (int64_t i = 0; i < numel; ++i) {
        float acc = load_as_f32(in[0], dtype, i);
        for (int r = 1; r < W; ++r) acc = acc + load_as_f32(in[r], dtype, i);
        store_from_f32(out, dtype, i, acc);
    }
    return 0;
}

/* all_gather_into_tensor, rank-major: bytes of in[r] land at r * numel
 * elements into out.  A byte copy: NaN payloads and every bit survive. */
int oracle_allgather_rank_major(const void *const *in, int W, int64_t numel, int esize, void *out)
{
    if (W < 1 || numel < 0 || !in || (esize != 2 && esize != 4)) return -1;
    if (numel == 0) return 0;
    if (!out) return -1;
    for (int r = 0; r < W; ++r) {
        if (!in[r]) return -1;
        memcpy((char *)out + (size_t)r * (size_t)numel * (size_t)esize, in[r],
               (size_t)numel * (size_t)esize);
    }
    return 0;
}

/* Param-contiguous allgather.  Each rank's shard is the concatenation of its
 * pieces of params 0..S-1, piece s holding E_s = splits[s] elements starting
 * at O_s = E_0 + ... + E_{s-1}.  Rank r's piece of param s lands at element
 * O_s * W + r * E_s of the output, so the output is param-major, then
 * rank-major inside each param. */
int oracle_allgather_param_contiguous(const void *const *in, int W, const int64_t *splits,
                                      int S, int esize, void *out)
{
    if (W < 1 || S < 0 || !in || (esize != 2 && esize != 4) || (S && !splits)) return -1;
    int64_t total = 0;
    for (int s = 0; s < S; ++s) {
        if (splits[s] < 0) return -1;
        total += splits[s];
    }
    if (total == 0) return 0;
    if (!out) return -1;
    for (int r = 0; r < W; ++r)
        if (!in[r]) return -1;
    int64_t O = 0;
    for (int s = 0; s < S; ++s) {
        int64_t E = splits[s];
        for (int r = 0; r < W; ++r)
            memcpy((char *)out + (size_t)(O * W + (int64_t)r * E) * (size_t)esize,
                   (const char *)in[r] + (size_t)O * (size_t)esize, (size_t)E * (size_t)esize);
        O += E;
    }
    return 0;
}

/* ------------------------------------------------------------ multi-threaded
 * The loops above, with the index range split over `threads` host threads
 * (<= 0: the OpenMP default).  Same per-element arithmetic, same order. */

/* Threads an *_mt call with threads <= 0 uses (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_allreduce_mt(const void *const *in, int W, int64_t numel, int dtype, void *out, int threads)
{
    if (W < 1 || numel < 0 || !in || elem_size(dtype) == 0) return -1;
    if (numel == 0) return 0;
    if (!out) return -1;
    for (int r = 0; r < W; ++r)
        if (!in[r]) return -1;
    if (threads <= 0) threads = oracle_max_threads();
    (void)threads;
    if (dtype == ORACLE_INT32) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads)
#endif
        for (int64_t i = 0; i < numel; ++i) {
            uint32_t acc = (uint32_t)((const int32_t *)in[0])[i];
            for (int r = 1; r < W; ++r) acc += (uint32_t)((const int32_t *)in[r])[i];
            ((uint32_t *)out)[i] = acc;
        }
        return 0;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(threads)
#endif
    for (int64_t i = 0; i < numel; ++i) {
        float acc = load_as_f32(in[0], dtype, i);
        for (int r = 1; r < W; ++r) acc = acc + load_as_f32(in[r], dtype, i);
        store_from_f32(out, dtype, i, acc);
    }
    return 0;
}

/* One byte-range copy of a gather, cut into 1 MiB pieces spread over threads. */
struct copy_piece {
    char *dst;
    const char *src;
    size_t len;
};

static void run_pieces(const struct copy_piece *c, int n, int threads)
{
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int i = 0; i < n; ++i) memcpy(c[i].dst, c[i].src, c[i].len);
}

#define ORACLE_PIECE ((size_t)1 << 20)

static int copy_ranges_mt(char *const *dst, const char *const *src, const size_t *len, int n, int threads)
{
    size_t pieces = 0;
    for (int i = 0; i < n; ++i) pieces += (len[i] + ORACLE_PIECE - 1) / ORACLE_PIECE;
    if (pieces == 0) return 0;
    if (pieces > (size_t)1 << 30) return -1;
    struct copy_piece buf[256];
    size_t k = 0;
    for (int i = 0; i < n; ++i)
        for (size_t o = 0; o < len[i]; o += ORACLE_PIECE) {
            buf[k].dst = dst[i] + o;
            buf[k].src = src[i] + o;
            buf[k].len = len[i] - o < ORACLE_PIECE ? len[i] - o : ORACLE_PIECE;
            if (++k == 256) {
                run_pieces(buf, 256, threads);
                k = 0;
            }
        }
    if (k) run_pieces(buf, (int)k, threads);
    return 0;
}

int oracle_allgather_rank_major_mt(const void *const *in, int W, int64_t numel, int esize, void *out,
                                   int threads)
{
    if (W < 1 || numel < 0 || !in || (esize != 2 && esize != 4)) return -1;
    if (numel == 0) return 0;
    if (!out) return -1;
    if (threads <= 0) threads = oracle_max_threads();
    for (int r = 0; r < W; ++r) {
        if (!in[r]) return -1;
        char *d = (char *)out + (size_t)r * (size_t)numel * (size_t)esize;
        const char *s = (const char *)in[r];
        size_t len = (size_t)numel * (size_t)esize;
        if (copy_ranges_mt(&d, &s, &len, 1, threads)) return -1;
    }
    return 0;
}

int oracle_allgather_param_contiguous_mt(const void *const *in, int W, const int64_t *splits, int S,
                                         int esize, void *out, int threads)
{
    if (W < 1 || S < 0 || !in || (esize != 2 && esize != 4) || (S && !splits)) return -1;
    int64_t total = 0;
    for (int s = 0; s < S; ++s) {
        if (splits[s] < 0) return -1;
        total += splits[s];
    }
    if (total == 0) return 0;
    if (!out) return -1;
    for (int r = 0; r < W; ++r)
        if (!in[r]) return -1;
    if (threads <= 0) threads = oracle_max_threads();
    int64_t O = 0;
    for (int s = 0; s < S; ++s) {
        int64_t E = splits[s];
        for (int r = 0; r < W; ++r) {
            char *d = (char *)out + (size_t)(O * W + (int64_t)r * E) * (size_t)esize;
            const char *src = (const char *)in[r] + (size_t)O * (size_t)esize;
            size_t len = (size_t)E * (size_t)esize;
            if (copy_ranges_mt(&d, &src, &len, 1, threads)) return -1;
        }
        O += E;
    }
    return 0;
}
