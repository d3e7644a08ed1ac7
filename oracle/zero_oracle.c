/*
 * zero_oracle.c -- plain, slow CPU oracle of the ZeRO-DP partitioned
 * mixed-precision optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only through the inputs the test generators
 * hand to both.
 *
 * Scalar loops, one element at a time, every floating-point operation written
 * out in the order of the method and rounded on its own (build with
 * -ffp-contract=off, never -ffast-math).
 *
 * Sources (page titles, sections):
 *  [notes]   "ZeRO: Memory Optimizations Toward Training Trillion Parameter
 *            Models" reading notes (papers.chlience.com): 5.1-5.4 memory
 *            formulas; 3 (Adam is coordinate-wise, so its state partitions);
 *            4 (all-reduce = reduce-scatter + all-gather, the averaged shard
 *            g_bar^(k) = (1/N_d) sum_r g_r^(k)); 7 and 9 (ZeRO-3 per-layer
 *            gather and gradient reduce-scatter).
 *  [stages]  "01 - ZeRO memory math and Stage 1/2" (DeepSpeed ZeRO stages
 *            1-2 walkthrough): 4 (1) flatten + pad to 2*world_size,
 *            4 (2) base = total // dp, remainder to the first ranks,
 *            4 (3) fp32 master copy of the own shard, 4 (4) parameter <->
 *            partition map, 6 (the step: overflow check, global norm,
 *            unscale+clip, Adam on the shard, copy back to 16 bit, all-gather).
 *  [paper]   "ZeRO: Memory Optimizations Toward Training Trillion Parameter
 *            Models" (Chinese translation), 3.1 (16 Psi accounting), 5.1-5.3
 *            (P_os, P_os+g, P_os+g+p and Figure 1's 7.5B example).
 *  [lecture] CMU 11-868 "Memory Optimization in Distributed Training" notes:
 *            slides 34-41 (reduce-scatter result converted to FP32, update,
 *            copy to FP16, all-gather), slide 64 (memory per stage).
 *
 * Readings taken where the pages leave a step open are listed beside the
 * function that takes them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================
 * 1. IEEE 754 conversions between binary32 and the 16-bit formats.
 *
 * Mixed precision keeps parameters and gradients in 16 bits and optimizer
 * states in 32 bits ([paper] 3.1; [stages] 1 table).  The formats:
 *   binary16 (fp16):  p = 11 significand bits, 5 exponent bits, bias 15
 *   bfloat16 (bf16):  p = 8  significand bits, 8 exponent bits, bias 127
 * Rounding is to nearest, ties to even (the IEEE default).
 * ====================================================================== */

static uint32_t f32_to_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }

/* Round the binary32 value x into a format with p significand bits and
 * ebits exponent bits.  Returns the 16-bit pattern.  Written from the
 * definition: x = sig * 2^(e-23) exactly; the target's quantum at x is
 * 2^(max(L, emin) - (p-1)) where L = floor(log2 |x|); divide, round half to
 * even, re-encode; a carry into the next binade and overflow past the largest
 * finite value (to infinity) fall out of the encoding step. */
static uint16_t round_to_narrow(float x, int p, int ebits)
{
    const uint32_t u = f32_to_bits(x);
    const uint32_t sign = u >> 31;
    const int e32 = (int)((u >> 23) & 0xffu);
    const uint32_t frac = u & 0x7fffffu;
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias;
    const uint32_t field_max = (1u << ebits) - 1u;
    const uint32_t sign_out = sign << (ebits + p - 1);

    if (e32 == 0xff) {
        if (frac == 0) return (uint16_t)(sign_out | (field_max << (p - 1)));          /* +-inf */
        return (uint16_t)(sign_out | (field_max << (p - 1)) | (1u << (p - 2)));      /* quiet NaN */
    }
    uint32_t sig;
    int e;                       /* x = sig * 2^(e - 23) */
    if (e32 == 0) { sig = frac; e = -126; } else { sig = frac | 0x800000u; e = e32 - 127; }
    if (sig == 0) return (uint16_t)sign_out;                                         /* +-0 */

    int top = 23;                /* position of the leading one of sig */
    while (!(sig & (1u << top))) top--;
    const int L = e - 23 + top;  /* floor(log2 |x|) */
    int Q = (L > emin ? L : emin) - (p - 1);   /* exponent of the target quantum */
    const int sh = Q - (e - 23);               /* x / 2^Q = sig / 2^sh */

    uint32_t q;
    if (sh <= 0) {
        q = sig << (-sh);                      /* exact (cannot happen for p < 24) */
    } else if (sh >= 25) {
        q = 0;                                 /* sig / 2^sh < 1/2 */
    } else {
        q = sig >> sh;
        const uint32_t rem = sig & ((1u << sh) - 1u);
        const uint32_t half = 1u << (sh - 1);
        if (rem > half || (rem == half && (q & 1u))) q++;
    }
    if (q == 0) return (uint16_t)sign_out;
    if (q == (1u << p)) { q >>= 1; Q += 1; }   /* rounded up into the next binade */
    if (q >= (1u << (p - 1))) {                /* normal */
        const int E = Q + (p - 1);
        const int field = E + bias;
        if (field >= (int)field_max) return (uint16_t)(sign_out | (field_max << (p - 1)));  /* overflow */
        return (uint16_t)(sign_out | ((uint32_t)field << (p - 1)) | (q - (1u << (p - 1))));
    }
    return (uint16_t)(sign_out | q);           /* subnormal: exponent field 0 */
}

static float widen_from_narrow(uint16_t h, int p, int ebits)
{
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t field_max = (1u << ebits) - 1u;
    const uint32_t sign = (uint32_t)h >> (ebits + p - 1);
    const uint32_t field = ((uint32_t)h >> (p - 1)) & field_max;
    const uint32_t mant = (uint32_t)h & ((1u << (p - 1)) - 1u);
    float v;
    if (field == field_max) v = mant ? NAN : INFINITY;
    else if (field == 0) v = ldexpf((float)mant, 1 - bias - (p - 1));
    else v = ldexpf((float)(mant | (1u << (p - 1))), (int)field - bias - (p - 1));
    return sign ? -v : v;
}

uint16_t orc_f32_to_f16(float x) { return round_to_narrow(x, 11, 5); }
uint16_t orc_f32_to_bf16(float x) { return round_to_narrow(x, 8, 8); }
float orc_f16_to_f32(uint16_t h) { return widen_from_narrow(h, 11, 5); }
float orc_bf16_to_f32(uint16_t h) { return widen_from_narrow(h, 8, 8); }

/* dtype codes used by this file: 1 = fp16, 2 = bf16 */
static float to_f32(uint16_t h, int dt) { return dt == 2 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h); }
static uint16_t from_f32(float x, int dt) { return dt == 2 ? orc_f32_to_bf16(x) : orc_f32_to_f16(x); }

void orc_round_array(const float* x, uint16_t* out, int64_t n, int dt)
{
    for (int64_t i = 0; i < n; i++) out[i] = from_f32(x[i], dt);
}

void orc_widen_array(const uint16_t* h, float* out, int64_t n, int dt)
{
    for (int64_t i = 0; i < n; i++) out[i] = to_f32(h[i], dt);
}

/* ======================================================================
 * 2. Exact accumulator for the sum of squares.
 *
 * The global gradient norm is a sum of per-shard sums of squares combined
 * by an all-reduce ([stages] 6, step 2).  The oracle sums exactly (a long
 * fixed-point accumulator) and rounds once, so its value does not depend on
 * the order of the terms or on how the vector was partitioned; that is what
 * lets the partitioned step and the unpartitioned one agree bit for bit.
 * Terms are non-negative doubles (squares of 16-bit values, exact in fp64).
 * ====================================================================== */

#define ACC_DIGITS 72          /* 32-bit digits: bit positions 0 .. 2303 */
#define ACC_OFFSET 1152        /* bit position of 2^0 (the lowest bit of a subnormal
                                  double, 2^-1126 after frexp scaling, lands at 26) */

typedef struct {
    int64_t d[ACC_DIGITS];     /* digit i holds a multiple of 2^(32 i - ACC_OFFSET) */
    int64_t adds;              /* additions since the last carry propagation */
    int32_t nonfinite;         /* a non-finite term was seen */
    int32_t pad;
} orc_acc;

int64_t orc_acc_size(void) { return (int64_t)sizeof(orc_acc); }

void orc_acc_clear(orc_acc* a) { memset(a, 0, sizeof *a); }

static void acc_normalize(orc_acc* a)
{
    int64_t carry = 0;
    for (int i = 0; i < ACC_DIGITS; i++) {
        const int64_t t = a->d[i] + carry;
        a->d[i] = t & 0xffffffffLL;
        carry = t >> 32;          /* all digits stay non-negative */
    }
    a->adds = 0;
}

void orc_acc_add(orc_acc* a, double x)
{
    if (!isfinite(x)) { a->nonfinite = 1; return; }
    if (x == 0.0) return;
    int ex;
    const double fr = frexp(x, &ex);                     /* x = fr * 2^ex, fr in [0.5, 1) */
    const uint64_t M = (uint64_t)ldexp(fr, 53);          /* 53-bit integer */
    const int pos = ex - 53 + ACC_OFFSET;                /* bit position of M's lowest bit */
    const int i = pos / 32, s = pos % 32;
    const uint64_t lo = M & 0xffffffffULL, hi = M >> 32; /* hi < 2^21 */
    const uint64_t l = lo << s, h = hi << s;             /* each < 2^64 */
    a->d[i]     += (int64_t)(l & 0xffffffffULL);
    a->d[i + 1] += (int64_t)(l >> 32) + (int64_t)(h & 0xffffffffULL);
    a->d[i + 2] += (int64_t)(h >> 32);
    if (++a->adds >= (1LL << 29)) acc_normalize(a);
}

void orc_acc_merge(orc_acc* a, const orc_acc* b)
{
    orc_acc c = *b;
    acc_normalize(&c);
    acc_normalize(a);
    for (int i = 0; i < ACC_DIGITS; i++) a->d[i] += c.d[i];
    a->nonfinite |= c.nonfinite;
    acc_normalize(a);
}

static int acc_bit(const orc_acc* a, int pos)
{
    if (pos < 0) return 0;
    return (int)((a->d[pos / 32] >> (pos % 32)) & 1);
}

/* Round the exact sum to the nearest double, ties to even. */
double orc_acc_value(const orc_acc* ain)
{
    orc_acc a = *ain;
    if (a.nonfinite) return INFINITY;
    acc_normalize(&a);
    int h = ACC_DIGITS - 1;
    while (h >= 0 && a.d[h] == 0) h--;
    if (h < 0) return 0.0;
    int b = 31;
    while (!((a.d[h] >> b) & 1)) b--;
    const int P = 32 * h + b;                         /* leading bit */
    int lsb = P - 52;
    if (lsb < -1074 + ACC_OFFSET) lsb = -1074 + ACC_OFFSET;
    uint64_t mant = 0;
    for (int k = P; k >= lsb; k--) mant = (mant << 1) | (uint64_t)acc_bit(&a, k);
    const int rbit = acc_bit(&a, lsb - 1);
    int sticky = 0;
    for (int k = lsb - 2; k >= 0 && !sticky; k--) sticky = acc_bit(&a, k);
    if (rbit && (sticky || (mant & 1u))) mant++;
    return ldexp((double)mant, lsb - ACC_OFFSET);     /* ldexp overflows to inf by itself */
}

/* Exact sum of an array of non-negative doubles (used to pin the accumulator). */
double orc_exact_sum(const double* x, int64_t n)
{
    orc_acc a;
    orc_acc_clear(&a);
    for (int64_t i = 0; i < n; i++) orc_acc_add(&a, x[i]);
    return orc_acc_value(&a);
}

/* ======================================================================
 * 3. Partition plan ([stages] 4 (1), (2), (4); 7 "alignment padding").
 *
 * Flatten: the group's tensors are laid end to end in declaration order.
 * mode 0 (the walkthrough's rule): pad the flat length to a multiple of
 *   2 * world_size, then split with base = total // dp and the remainder to
 *   the first ranks (the remainder is then 0; padding sits at the tail of
 *   the last rank).
 * mode 1: the same base/remainder rule applied to the unpadded length.
 * ====================================================================== */

int orc_plan(const int64_t* numels, int n, int ws, int mode,
             int64_t* tensor_offsets, int64_t* rank_offsets, int64_t* rank_numels,
             int64_t* padded_total, int64_t* padding)
{
    if (n < 0 || ws < 1 || (mode != 0 && mode != 1)) return -1;
    int64_t total = 0;
    for (int i = 0; i < n; i++) {
        if (numels[i] < 0) return -1;
        tensor_offsets[i] = total;
        total += numels[i];
    }
    int64_t flat = total;
    if (mode == 0) {
        const int64_t align = 2 * (int64_t)ws;
        flat = ((total + align - 1) / align) * align;
    }
    const int64_t base = flat / ws, remaining = flat % ws;
    int64_t off = 0;
    for (int r = 0; r < ws; r++) {
        rank_offsets[r] = off;
        rank_numels[r] = base + (r < remaining ? 1 : 0);
        off += rank_numels[r];
    }
    *padded_total = flat;
    *padding = flat - total;
    return 0;
}

/* For one rank: every tensor that overlaps its shard, as
 * (tensor index, first element inside the tensor, first element inside the
 * shard, length).  Returns the number of rows written to out[4*k]. */
int orc_plan_intersections(const int64_t* tensor_offsets, const int64_t* numels, int n,
                           int64_t rank_offset, int64_t rank_numel, int64_t* out)
{
    int k = 0;
    const int64_t lo = rank_offset, hi = rank_offset + rank_numel;
    for (int i = 0; i < n; i++) {
        const int64_t a = tensor_offsets[i], b = tensor_offsets[i] + numels[i];
        const int64_t s = a > lo ? a : lo, e = b < hi ? b : hi;
        if (e > s) {
            out[4 * k + 0] = i;
            out[4 * k + 1] = s - a;
            out[4 * k + 2] = s - lo;
            out[4 * k + 3] = e - s;
            k++;
        }
    }
    return k;
}

/* ======================================================================
 * 4. Memory model ([paper] 5.1-5.3 and Figure 1; [notes] 5.1-5.4;
 *    [lecture] slide 64).  Bytes of model states per device:
 *      stage 0 (DP):        (4 + K) Psi
 *      stage 1 (P_os):      4 Psi + K Psi / N_d
 *      stage 2 (P_os+g):    2 Psi + (K + 2) Psi / N_d
 *      stage 3 (P_os+g+p):  (4 + K) Psi / N_d
 * ====================================================================== */

double orc_mem_model(double psi, double K, int nd, int stage)
{
    const double N = (double)nd;
    switch (stage) {
    case 0: return (4.0 + K) * psi;
    case 1: return 4.0 * psi + K * psi / N;
    case 2: return 2.0 * psi + (K + 2.0) * psi / N;
    case 3: return (4.0 + K) * psi / N;
    default: return -1.0;
    }
}

/* Plan-exact model states of one rank, with temporaries.  The stage
 * formulas above take a rank's share as Psi / N_d; here each term takes the
 * plan's own sizes: F = elements of a 16-bit flat buffer the stage keeps
 * whole (the padded total; Psi for stage 0), n = the rank's shard.  Which
 * buffers a stage keeps whole and which it partitions follows [paper]
 * 5.1-5.3: P_os partitions the optimizer states, P_os+g the gradients too,
 * P_os+g+p the parameters too.  `sets` copies of the optimizer state are
 * held (2 when the state is double-buffered).  The temporaries are the
 * fp32 fused flat buffer of [paper] 3.2 and 6.2 (4 bytes an element) and
 * 16-bit buffers (2 bytes an element).
 * out[0] parameters, out[1] gradients, out[2] optimizer states,
 * out[3] temporaries, out[4] their sum.  Returns 0, or -1 on a bad argument. */
int orc_mem_model_plan(int64_t F, int64_t n, double K, int stage, int sets,
                       int64_t fp32_temp, int64_t b16_temp, double* out)
{
    if (F < 0 || n < 0 || K < 0.0 || stage < 0 || stage > 3 || sets < 1 ||
        fp32_temp < 0 || b16_temp < 0)
        return -1;
    const double params_whole = (stage <= 2) ? (double)F : (double)n;
    const double grads_whole = (stage <= 1) ? (double)F : (double)n;
    const double states_of = (stage == 0) ? (double)F : (double)n;
    out[0] = 2.0 * params_whole;
    out[1] = 2.0 * grads_whole;
    out[2] = K * states_of * (double)sets;
    out[3] = 4.0 * (double)fp32_temp + 2.0 * (double)b16_temp;
    out[4] = out[0] + out[1] + out[2] + out[3];
    return 0;
}

/* ======================================================================
 * 5. The step.
 * ====================================================================== */

/* Host scalars of one AdamW step, each computed in fp64 from the fp32
 * hyper-parameters and rounded once to fp32.
 * Adam per coordinate ([notes] 3):  m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
 * theta <- theta - lr * m_hat / (sqrt(v_hat) + eps).  Reading: m_hat, v_hat are
 * the usual bias corrections m/(1-b1^t), v/(1-b2^t); weight decay is decoupled
 * (theta <- theta (1 - lr wd) before the Adam update).  The corrections are
 * folded into two scalars: ss = lr/(1-b1^t) and rb2 = 1/sqrt(1-b2^t), so that
 * the update reads theta - ss * m / (sqrt(v) rb2 + eps) -- the same quantity. */
typedef struct {
    float b1, b2, omb1, omb2, eps, wdf, ss, rb2;
} orc_scalars;

void orc_make_scalars(float lr, float beta1, float beta2, float eps, float wd, int64_t t,
                      orc_scalars* s)
{
    const double bc1 = 1.0 - pow((double)beta1, (double)t);
    const double bc2 = 1.0 - pow((double)beta2, (double)t);
    s->b1 = beta1;
    s->b2 = beta2;
    s->omb1 = (float)(1.0 - (double)beta1);
    s->omb2 = (float)(1.0 - (double)beta2);
    s->eps = eps;
    s->wdf = (float)(1.0 - (double)lr * (double)wd);
    s->ss = (float)((double)lr / bc1);
    s->rb2 = (float)(1.0 / sqrt(bc2));
}

/* Unscale and clip ([stages] 6, step 3).  norm = sqrt(sumsq) / S is the true
 * gradient norm; reading: when clipping is on (max_norm > 0) the coefficient is
 * c = max_norm / (norm + 1e-6), applied only when it is below 1.  The single
 * multiplier applied to the scaled gradient is k = fp32(c / S). */
float orc_grad_multiplier(double sumsq, double loss_scale, double max_norm, double* norm_out,
                          double* clip_out)
{
    const double norm = sqrt(sumsq) / loss_scale;
    double c = 1.0;
    if (max_norm > 0.0) {
        const double cc = max_norm / (norm + 1e-6);
        if (cc < 1.0) c = cc;
    }
    if (norm_out) *norm_out = norm;
    if (clip_out) *clip_out = c;
    return (float)(c / loss_scale);
}

/* AdamW on one fp32 coordinate, every operation rounded to fp32, in the order
 * of the update rule above.  a is the averaged 16-bit gradient (still scaled),
 * widened to fp32; k unscales (and clips) it. */
static void adamw_one(float* theta, float* m, float* v, float a, float k, const orc_scalars* s)
{
    const float g = a * k;
    float th = *theta * s->wdf;
    const float mm = s->b1 * *m + s->omb1 * g;
    const float g2 = g * g;
    const float vv = s->b2 * *v + s->omb2 * g2;
    const float den = sqrtf(vv) * s->rb2 + s->eps;
    const float upd = mm / den;
    th = th - s->ss * upd;
    *theta = th;
    *m = mm;
    *v = vv;
}

/* The reduce-scatter's arithmetic for one element ([notes] 4:
 * g_bar = (1/N_d) sum_r g_r).  Reading: the N_d 16-bit values are widened to
 * fp32 and summed in rank order 0..N_d-1, divided by N_d in fp32, and the
 * average is rounded once to the gradient dtype -- the reduced shard is still
 * a 16-bit gradient that is converted to FP32 afterwards ([lecture] slides
 * 34-35). */
static uint16_t reduce_one(const uint16_t* const* slices, int n_slices, int64_t idx, int gdt)
{
    float s = 0.0f;
    for (int r = 0; r < n_slices; r++) s = s + to_f32(slices[r][idx], gdt);
    return from_f32(s / (float)n_slices, gdt);
}

/* Reduce `numel` elements starting at `off` in every slice into out (16-bit). */
void orc_reduce(const uint16_t* const* slices, int n_slices, int gdt, int64_t off, int64_t numel,
                uint16_t* out)
{
    for (int64_t j = 0; j < numel; j++) out[j] = reduce_one(slices, n_slices, off + j, gdt);
}

/* Overflow and sum of squares over already-reduced 16-bit gradients
 * ([stages] 6, steps 1-2): a value is an overflow when it is inf or NaN;
 * squares are taken of the fp32 widening, in fp64 (exact). */
void orc_stats(const uint16_t* a, int64_t numel, int gdt, orc_acc* acc, int32_t* overflow)
{
    for (int64_t j = 0; j < numel; j++) {
        const float x = to_f32(a[j], gdt);
        if (!isfinite(x)) { *overflow = 1; acc->nonfinite = 1; continue; }
        orc_acc_add(acc, (double)x * (double)x);
    }
}

/* Reduce and take the statistics in one sweep, without keeping the reduced
 * values (used to get the global norm of full-size workloads chunk by chunk). */
void orc_reduce_stats(const uint16_t* const* slices, int n_slices, int gdt, int64_t off,
                      int64_t numel, orc_acc* acc, int32_t* overflow)
{
    for (int64_t j = 0; j < numel; j++) {
        const uint16_t a = reduce_one(slices, n_slices, off + j, gdt);
        orc_stats(&a, 1, gdt, acc, overflow);
    }
}

/* AdamW + cast-store for n elements given their reduced gradients: the
 * master/m/v arrays are updated in place and param[j] = round_P(theta_j)
 * ([stages] 6, steps 4-5; [lecture] slides 36-40). */
void orc_apply(const uint16_t* a, int gdt, float* master, float* m, float* v, int64_t n,
               uint16_t* param, int pdt, float k, const orc_scalars* s)
{
    for (int64_t j = 0; j < n; j++) {
        adamw_one(&master[j], &m[j], &v[j], to_f32(a[j], gdt), k, s);
        param[j] = from_f32(master[j], pdt);
    }
}

typedef struct {
    int32_t overflow;    /* any reduced gradient element (or the other ranks') was inf/NaN */
    int32_t applied;     /* 1 when the update was made; 0 when the step was skipped */
    double sumsq;        /* sum of squares of the scaled reduced gradient, incl. extra_sumsq */
    double grad_norm;    /* sqrt(sumsq) / loss_scale */
    double clip_coef;    /* c (1 when not clipping) */
    float grad_mult;     /* k = fp32(c / loss_scale) */
    float pad;
} orc_result;

/* One partitioned step over n_shards shards that share the call's global
 * decisions (all simulated ranks, or one rank plus the other ranks'
 * contributions given as extra_sumsq / extra_overflow -- the scalar
 * all-reduce of the norm).  Order of [stages] 6:
 *   reduce each shard's slices -> overflow check (skip on overflow: nothing
 *   changes) -> global norm -> unscale + clip -> AdamW on the fp32 shard ->
 *   copy the result to 16 bits at the shard's offset in the flat buffer (the
 *   all-gather destination, shared by every simulated rank).
 * Slice element of shard s, rank r, element j: slices[r][grad_off[s] + j].
 * grad_out[s] (optional) receives the reduced 16-bit shard. */
int orc_zero_step(const uint16_t* const* slices, int n_slices, int gdt,
                  int n_shards, const int64_t* numel, const int64_t* grad_off,
                  const int64_t* param_off,
                  float* const* master, float* const* m, float* const* v,
                  uint16_t* flat_param, int pdt,
                  float lr, float beta1, float beta2, float eps, float wd, float max_norm,
                  int64_t t, double loss_scale, double extra_sumsq, int extra_overflow,
                  uint16_t* const* grad_out, orc_result* res)
{
    uint16_t** red = (uint16_t**)calloc((size_t)(n_shards > 0 ? n_shards : 1), sizeof(uint16_t*));
    if (!red) return -1;
    orc_acc acc;
    orc_acc_clear(&acc);
    int32_t ovf = extra_overflow ? 1 : 0;
    int rc = 0;
    for (int s = 0; s < n_shards; s++) {
        red[s] = (uint16_t*)malloc((size_t)(numel[s] > 0 ? numel[s] : 1) * sizeof(uint16_t));
        if (!red[s]) { rc = -1; goto done; }
        orc_reduce(slices, n_slices, gdt, grad_off[s], numel[s], red[s]);
        orc_stats(red[s], numel[s], gdt, &acc, &ovf);
        if (grad_out && grad_out[s]) memcpy(grad_out[s], red[s], (size_t)numel[s] * sizeof(uint16_t));
    }
    {
        const double own = orc_acc_value(&acc);
        res->overflow = ovf;
        res->sumsq = own + extra_sumsq;
        double norm, clip;
        const float k = orc_grad_multiplier(res->sumsq, loss_scale, (double)max_norm, &norm, &clip);
        res->grad_norm = norm;
        res->clip_coef = clip;
        res->grad_mult = k;
        res->pad = 0.0f;
        if (ovf) { res->applied = 0; goto done; }
        orc_scalars sc;
        orc_make_scalars(lr, beta1, beta2, eps, wd, t, &sc);
        for (int s = 0; s < n_shards; s++)
            orc_apply(red[s], gdt, master[s], m[s], v[s], numel[s], flat_param + param_off[s], pdt, k,
                      &sc);
        res->applied = 1;
    }
done:
    for (int s = 0; s < n_shards; s++) free(red[s]);
    free(red);
    return rc;
}

/* The unpartitioned data-parallel step the ZeRO step must reproduce
 * ([notes] 6 and 9, "standard DP"): every rank all-reduces the whole gradient
 * (the average over ranks of every coordinate) and runs the same full AdamW
 * on the whole fp32 vector, then copies it to 16 bits.  Here one copy of that
 * computation over all n elements of the flat vector. */
int orc_ddp_step(const uint16_t* const* grads, int n_ranks, int gdt, int64_t n,
                 float* master, float* m, float* v, uint16_t* param, int pdt,
                 float lr, float beta1, float beta2, float eps, float wd, float max_norm,
                 int64_t t, double loss_scale, orc_result* res)
{
    uint16_t* avg = (uint16_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(uint16_t));
    if (!avg) return -1;
    orc_acc acc;
    orc_acc_clear(&acc);
    int32_t ovf = 0;
    orc_reduce(grads, n_ranks, gdt, 0, n, avg);
    orc_stats(avg, n, gdt, &acc, &ovf);
    res->overflow = ovf;
    res->sumsq = orc_acc_value(&acc);
    double norm, clip;
    const float k = orc_grad_multiplier(res->sumsq, loss_scale, (double)max_norm, &norm, &clip);
    res->grad_norm = norm;
    res->clip_coef = clip;
    res->grad_mult = k;
    res->pad = 0.0f;
    res->applied = 0;
    if (!ovf) {
        orc_scalars sc;
        orc_make_scalars(lr, beta1, beta2, eps, wd, t, &sc);
        orc_apply(avg, gdt, master, m, v, n, param, pdt, k, &sc);
        res->applied = 1;
    }
    free(avg);
    return 0;
}

/* ======================================================================
 * 6. ZeRO-3 per-layer steps ([notes] 7 and 9, stage 3; [paper] 7.2.2).
 * A layer (unit) of U elements is split into N equal parts; rank r keeps
 * part r.  Before the layer's forward, and again before its backward, the
 * parts are gathered into one contiguous layer buffer:
 *     layer[r * U/N + j] = part_r[j].
 * After the backward, the owner of part o receives the average of every
 * rank's gradient for its part (the reduce-scatter, same arithmetic as
 * reduce_one above).
 * ====================================================================== */

void orc_zero3_gather(const uint16_t* const* parts, int n, int64_t part_numel, uint16_t* layer)
{
    for (int r = 0; r < n; r++)
        for (int64_t j = 0; j < part_numel; j++) layer[(int64_t)r * part_numel + j] = parts[r][j];
}

void orc_zero3_reduce(const uint16_t* const* buckets, int n, int owner, int64_t part_numel, int gdt,
                      uint16_t* grad_part, orc_acc* acc, int32_t* overflow)
{
    orc_reduce(buckets, n, gdt, (int64_t)owner * part_numel, part_numel, grad_part);
    orc_stats(grad_part, part_numel, gdt, acc, overflow);
}

/* ======================================================================
 * 7. Communication volume ([paper] 7.1-7.2; [notes] 4 and 5.5).
 * Elements one data-parallel rank sends (and receives) per step in the
 * data-parallel collectives.  A reduce-scatter or an all-gather of Psi
 * elements is counted as Psi ([paper] 7.1); with ring = 1 a ring moves
 * (N_d - 1)/N_d of that per phase ([notes] 4).
 *   stage 0 (DP): all-reduce = reduce-scatter + all-gather      2 phases
 *   stage 1, 2:   gradient reduce-scatter + parameter all-gather 2 phases
 *   stage 3:      parameter all-gather for the forward and again for the
 *                 backward, plus the gradient reduce-scatter     3 phases
 * ====================================================================== */

double orc_comm_volume(double psi, int nd, int stage, int ring)
{
    if (nd < 1 || stage < 0 || stage > 3) return -1.0;
    const double phase = ring ? psi * (double)(nd - 1) / (double)nd : psi;
    return (stage == 3 ? 3.0 : 2.0) * phase;
}

/* ======================================================================
 * 8. Round-robin order of a group's tensors ([stages] 4.1): before
 * flattening, tensor i is put in group i mod world_size and the groups are
 * laid out one after another, each in its original order, so that tensors
 * that are adjacent in the original (backward) order land in different
 * ranks' shards.  order[k] = original index of the tensor placed k-th.
 * ====================================================================== */

int orc_round_robin(int n, int ws, int64_t* order)
{
    if (n < 0 || ws < 1) return -1;
    int k = 0;
    for (int g = 0; g < ws; g++)
        for (int i = g; i < n; i += ws) order[k++] = i;
    return 0;
}

/* ======================================================================
 * 9. ZeRO-3 owner broadcast ([paper] 5.3 and 7.2.2): each rank keeps a
 * contiguous segment of the flat parameter vector; a layer is rebuilt from
 * the pieces of the owners' segments it spans, laid end to end.
 * ====================================================================== */

void orc_gather_segments(const uint16_t* const* segs, const int64_t* lens, int n, uint16_t* out)
{
    int64_t o = 0;
    for (int p = 0; p < n; p++)
        for (int64_t j = 0; j < lens[p]; j++) out[o++] = segs[p][j];
}
