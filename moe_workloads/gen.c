/*
 * Seeded synthetic inputs for the MoE prefill layer: token activations, router
 * logits / top-k routing, and quantized expert weights packed as expert records.
 *
 * This module holds input generation only, none of the layer's arithmetic.  Both
 * the CUDA library's tests and the CPU oracle's tests take their inputs from it.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) used as a counter-based hash: stream key
 *   key = splitmix64(seed ^ splitmix64(tensor_id)),
 * element i draws u64 = splitmix64(key + i).  A uniform is (u64 >> 11) * 2^-53.
 * Normals come in pairs (Box-Muller, in double, rounded to fp32): with
 * u0 = uniform 2p, u1 = uniform 2p+1 and r = sqrt(-2 ln(1 - u0)),
 *   normal 2p = r cos(2 pi u1),  normal 2p+1 = r sin(2 pi u1).
 * Results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static uint64_t splitmix64(uint64_t z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t gen_key(uint64_t seed, uint64_t tensor_id) { return splitmix64(seed ^ splitmix64(tensor_id)); }

static double uniform_at(uint64_t key, uint64_t i) {
    return (double)(splitmix64(key + i) >> 11) * 0x1.0p-53;
}

static double normal_at(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t p = i >> 1;
    double u0 = uniform_at(key, 2 * p), u1 = uniform_at(key, 2 * p + 1);
    double r = sqrt(-2.0 * log(1.0 - u0));
    return (i & 1) ? r * sin(two_pi * u1) : r * cos(two_pi * u1);
}

/* normals i and i+1 (i even) at the cost of one pair */
static void normal_pair(uint64_t key, uint64_t i, double* a, double* b) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t p = i >> 1;
    double u0 = uniform_at(key, 2 * p), u1 = uniform_at(key, 2 * p + 1);
    double r = sqrt(-2.0 * log(1.0 - u0));
    *a = r * cos(two_pi * u1);
    *b = r * sin(two_pi * u1);
}

/* out[i] = fp32(scale * normal(start + i)) for i < n, pairs at a time */
static void fill_normals(uint64_t key, uint64_t start, size_t lo, size_t hi, double scale, float* out) {
    size_t i = lo;
    if (i < hi && ((start + i) & 1)) {
        out[i] = (float)(scale * normal_at(key, start + i));
        ++i;
    }
    for (; i + 1 < hi; i += 2) {
        double a, b;
        normal_pair(key, start + i, &a, &b);
        out[i] = (float)(scale * a);
        out[i + 1] = (float)(scale * b);
    }
    if (i < hi) out[i] = (float)(scale * normal_at(key, start + i));
}

void gen_uniform_f64(uint64_t seed, uint64_t tensor_id, uint64_t start, size_t n, double* out) {
    uint64_t key = gen_key(seed, tensor_id);
    for (size_t i = 0; i < n; ++i) out[i] = uniform_at(key, start + i);
}

typedef struct {
    uint64_t key, start;
    size_t lo, hi;
    double scale;
    float* out;
} normal_job;

static void* normal_worker(void* p) {
    normal_job* j = (normal_job*)p;
    fill_normals(j->key, j->start, j->lo, j->hi, j->scale, j->out);
    return NULL;
}

/* out[i] = fp32(scale * N(0,1) draw number start+i of (seed, tensor_id)). */
void gen_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, size_t n, double scale,
                    float* out, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    pthread_t th[256];
    normal_job jobs[256];
    uint64_t key = gen_key(seed, tensor_id);
    for (int t = 0; t < threads; ++t) {
        jobs[t].key = key;
        jobs[t].start = start;
        jobs[t].lo = n * (size_t)t / (size_t)threads;
        jobs[t].hi = n * (size_t)(t + 1) / (size_t)threads;
        jobs[t].scale = scale;
        jobs[t].out = out;
        if (threads > 1) pthread_create(&th[t], NULL, normal_worker, &jobs[t]);
        else normal_worker(&jobs[t]);
    }
    if (threads > 1)
        for (int t = 0; t < threads; ++t) pthread_join(th[t], NULL);
}

/* ---------------- expert records (the library's weight format) --------------- */
/* gate [f x d], up [f x d], down [d x f]; per matrix: quant plane, fp16 d plane
   [K/32][rows] (block-major), Q4_1 also fp16 m plane [K/32][rows]; planes
   128-byte aligned.  Quant bytes per row: K (Q8_0), K/2 (Q4_1), K/4 (Q2_0, Q2_K).
   Q2_K (wtype 3, K a multiple of 256): 2-bit codes as Q2_0, fp16 d and dmin per
   256-weight super-block in planes [K/256][rows], and one byte per 16-weight
   sub-block, scale sc in the low and min mn in the high nibble, plane
   [K/16][rows]; w = d*sc*c - dmin*mn. */
static size_t a128(size_t x) { return (x + 127u) & ~(size_t)127u; }

static size_t mat_bytes4(int wtype, int rows, int k, size_t* qoff, size_t* doff, size_t* moff,
                         size_t* soff) {
    size_t qb = (size_t)rows * (size_t)k / (wtype == 1 ? 2u : (wtype == 2 || wtype == 3) ? 4u : 1u);
    size_t sb = (size_t)rows * (size_t)(k / (wtype == 3 ? 256 : 32)) * 2u;
    *qoff = 0;
    *doff = a128(qb);
    *moff = *doff + a128(sb);
    *soff = *moff + ((wtype == 1 || wtype == 3) ? a128(sb) : 0u);
    return *soff + (wtype == 3 ? a128((size_t)rows * (size_t)(k / 16)) : 0u);
}

static size_t mat_bytes(int wtype, int rows, int k, size_t* qoff, size_t* doff, size_t* moff) {
    size_t soff;
    return mat_bytes4(wtype, rows, k, qoff, doff, moff, &soff);
}

size_t gen_record_bytes(int wtype, int d, int f) {
    size_t a, b, c;
    return 2u * mat_bytes(wtype, f, d, &a, &b, &c) + mat_bytes(wtype, d, f, &a, &b, &c);
}

static uint16_t to_f16_bits(float v) {
    _Float16 h = (_Float16)v; /* IEEE round to nearest even */
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static float from_f16_bits(uint16_t b) {
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

/* Q2_K: one 256-weight super-block v of a row.  Per 16-weight sub-block j the
   codes cover [-mn_j, max_j] in 3 steps; the super-block stores d = max step / 15
   and dmin = max mn_j / 15 (fp16), each sub-block sc_j = round(step_j / d) and
   mn_j = round(mn_j / dmin) in [0, 15], and c = round((w + dmin*mn) / (d*sc)) in
   [0, 3] from the stored (rounded) values. */
static void pack_q2k_super(const float* v, uint8_t* codes, uint8_t* scmn, int rows, int r,
                           int sb, uint16_t* dp, uint16_t* mp) {
    float step[16], mins[16];
    float smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float lo = v[16 * j], hi = v[16 * j];
        for (int i = 1; i < 16; ++i) {
            lo = fminf(lo, v[16 * j + i]);
            hi = fmaxf(hi, v[16 * j + i]);
        }
        mins[j] = fmaxf(0.0f, -lo);
        step[j] = (hi + mins[j]) / 3.0f;
        smax = fmaxf(smax, step[j]);
        mmax = fmaxf(mmax, mins[j]);
    }
    const uint16_t dbits = to_f16_bits(smax / 15.0f), mbits = to_f16_bits(mmax / 15.0f);
    const float dd = from_f16_bits(dbits), dm = from_f16_bits(mbits);
    dp[(size_t)sb * rows + r] = dbits;
    mp[(size_t)sb * rows + r] = mbits;
    for (int j = 0; j < 16; ++j) {
        int sc = dd > 0.0f ? (int)fminf(15.0f, fmaxf(0.0f, roundf(step[j] / dd))) : 0;
        int mn = dm > 0.0f ? (int)fminf(15.0f, fmaxf(0.0f, roundf(mins[j] / dm))) : 0;
        scmn[((size_t)sb * 16 + j) * rows + r] = (uint8_t)(sc | (mn << 4));
        const float s = dd * (float)sc, m = dm * (float)mn;
        for (int q4 = 0; q4 < 4; ++q4) {  /* four bytes of four codes each */
            uint8_t byte = 0;
            for (int i = 0; i < 4; ++i) {
                const float x = v[16 * j + 4 * q4 + i];
                int c = s > 0.0f ? (int)fminf(3.0f, fmaxf(0.0f, roundf((x + m) / s))) : 0;
                byte |= (uint8_t)(c << (2 * i));
            }
            codes[16 * j / 4 + q4] = byte;
        }
    }
}

/* Quantize one matrix of weights w [rows x k] into the record at dst. */
static void pack_matrix(int wtype, const float* w, int rows, int k, uint8_t* dst) {
    size_t qo, dof, mo, so;
    mat_bytes4(wtype, rows, k, &qo, &dof, &mo, &so);
    if (wtype == 3) {
        for (int r = 0; r < rows; ++r)
            for (int sb = 0; sb < k / 256; ++sb)
                pack_q2k_super(w + (size_t)r * k + (size_t)sb * 256,
                               dst + qo + (size_t)r * (k / 4) + (size_t)sb * 64, dst + so, rows, r, sb,
                               (uint16_t*)(dst + dof), (uint16_t*)(dst + mo));
        return;
    }
    uint8_t* qp = dst + qo;
    uint16_t* dp = (uint16_t*)(dst + dof);
    uint16_t* mp = (uint16_t*)(dst + mo);
    int nb = k / 32;
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            const float* v = w + (size_t)r * k + (size_t)b * 32;
            if (wtype == 0) { /* Q8_0: d = amax/127, q = round(w/d) */
                float amax = 0.0f;
                for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                float dd = amax / 127.0f;
                int8_t* q = (int8_t*)qp + (size_t)r * k + (size_t)b * 32;
                for (int i = 0; i < 32; ++i) {
                    float x = dd > 0.0f ? roundf(v[i] / dd) : 0.0f;
                    x = fminf(127.0f, fmaxf(-127.0f, x));
                    q[i] = (int8_t)x;
                }
                dp[(size_t)b * rows + r] = to_f16_bits(dd);
            } else if (wtype == 2) { /* Q2_0: d = amax/2, c = round(w/d) + 2 in [0,3] */
                float amax = 0.0f;
                for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
                float dd = amax / 2.0f;
                uint8_t* q = qp + (size_t)r * (k / 4) + (size_t)b * 8;
                for (int j = 0; j < 8; ++j) {
                    uint8_t byte = 0;
                    for (int i = 0; i < 4; ++i) {
                        float x = dd > 0.0f ? roundf(v[4 * j + i] / dd) : 0.0f;
                        x = fminf(1.0f, fmaxf(-2.0f, x));
                        byte |= (uint8_t)(((int)x + 2) << (2 * i));
                    }
                    q[j] = byte;
                }
                dp[(size_t)b * rows + r] = to_f16_bits(dd);
            } else { /* Q4_1: d = (max-min)/15, m = min, q = round((w-m)/d) in [0,15] */
                float mn = v[0], mx = v[0];
                for (int i = 1; i < 32; ++i) {
                    mn = fminf(mn, v[i]);
                    mx = fmaxf(mx, v[i]);
                }
                float dd = (mx - mn) / 15.0f;
                uint8_t* q = qp + (size_t)r * (k / 2) + (size_t)b * 16;
                for (int j = 0; j < 16; ++j) {
                    int lo = 0, hi = 0;
                    if (dd > 0.0f) {
                        lo = (int)fminf(15.0f, fmaxf(0.0f, roundf((v[2 * j] - mn) / dd)));
                        hi = (int)fminf(15.0f, fmaxf(0.0f, roundf((v[2 * j + 1] - mn) / dd)));
                    }
                    q[j] = (uint8_t)(lo | (hi << 4));
                }
                dp[(size_t)b * rows + r] = to_f16_bits(dd);
                mp[(size_t)b * rows + r] = to_f16_bits(mn);
            }
        }
    }
}

typedef struct {
    int wtype, d, f, e0, e1;
    uint64_t seed;
    double sigma;
    uint8_t* arena;
    size_t stride;
} rec_job;

static void* rec_worker(void* p) {
    rec_job* j = (rec_job*)p;
    size_t maxel = (size_t)j->f * (size_t)j->d;
    float* w = (float*)malloc(maxel * sizeof(float));
    size_t qo, dof, mo;
    size_t gbytes = mat_bytes(j->wtype, j->f, j->d, &qo, &dof, &mo);
    for (int e = j->e0; e < j->e1; ++e) {
        uint8_t* rec = j->arena + (size_t)e * j->stride;
        for (int m = 0; m < 3; ++m) {
            int rows = m < 2 ? j->f : j->d, k = m < 2 ? j->d : j->f;
            uint64_t key = gen_key(j->seed, 100u + 3u * (uint64_t)e + (uint64_t)m);
            fill_normals(key, 0, 0, maxel, j->sigma, w);
            pack_matrix(j->wtype, w, rows, k, rec + (size_t)m * gbytes);
        }
    }
    free(w);
    return NULL;
}

/* Fill E expert records (arena_stride bytes apart) with N(0, sigma) weights,
   quantized to wtype (0 = Q8_0, 1 = Q4_1, 2 = Q2_0, 3 = Q2_K).  Expert e, matrix m (gate, up,
   down) draws from tensor id 100 + 3e + m, element index row*k + col. */
void gen_expert_records(int wtype, int E, int d, int f, uint64_t seed, double sigma,
                        uint8_t* arena, size_t arena_stride, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (threads > E) threads = E > 0 ? E : 1;
    pthread_t th[256];
    rec_job jobs[256];
    for (int t = 0; t < threads; ++t) {
        rec_job j = {wtype, d, f, E * t / threads, E * (t + 1) / threads, seed, sigma, arena,
                     arena_stride};
        jobs[t] = j;
        if (threads > 1) pthread_create(&th[t], NULL, rec_worker, &jobs[t]);
        else rec_worker(&jobs[t]);
    }
    if (threads > 1)
        for (int t = 0; t < threads; ++t) pthread_join(th[t], NULL);
}
