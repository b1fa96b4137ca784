/*
 * oracle.c -- plain, single-threaded CPU oracle for the deterministic
 * multi-writer reduction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The GPU library
 * shares no code, header, table or helper with it, and neither includes the
 * other.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off matters: without it GCC (on aarch64 by default) may fuse
 * a product and the following add into one FMA, which rounds once instead of
 * twice and changes the bits this oracle is meant to fix.
 *
 * What is computed (sources, in the words of the pages):
 *  - Floating-point addition is not associative; every add rounds to nearest,
 *    so changing the order changes the last bits ("DeepSeek-V4 book, Ch 09,
 *    Batch invariance and determinism", section 1 and its BF16 worked example).
 *  - The MoE token combine/unpermute adds each permuted row into its token's
 *    output row: out.index_add_(0, sorted_indices, permuted_tokens) is the
 *    deterministic branch, scatter_add_ the atomic one ("Megatron-LM
 *    determinism developer reference", section 3.1, op catalog).
 *  - Several writers to one address get private slots that are merged in a
 *    fixed order ("Bit-exact training interview notes", table "where
 *    nondeterminism comes from", multi-writer row); every EP size must go
 *    through the same fp32 reduction tree (same page, "why pay the overhead",
 *    EP-size-invariant expert combine).
 *  - The MoE backward orders tokens by (expert id, original token id) and
 *    merges in that sorted order (Ch 09, section 3.2); the mHC backward sums
 *    per-split buffers in split-id order (Ch 09, section 3.3).
 *
 * The pages fix the problem but print no tree, so this library fixes one
 * canonical order and the oracle writes it out literally:
 *   1. the terms of destination m are the sources i with idx[i] = m, taken in
 *      ascending order key (src_id[i], default i);
 *   2. term j is p_j = fl32(w[i_j] * fl32(x[i_j][h])) -- one binary32 multiply,
 *      round to nearest even; no multiply when w is absent;
 *   3. chunks of 32 consecutive terms are folded left to right, the fold
 *      starting from the chunk's first term (never from 0.0);
 *   4. the chunk sums form level 0 of a level-wise pairwise tree:
 *      L[t+1][k] = L[t][2k] + L[t][2k+1]; when L[t] has odd length its last
 *      element is carried up unchanged; repeat until one value remains;
 *   5. an empty destination is +0.0;
 *   6. the result is stored as binary32, or rounded to bf16 (nearest even).
 * The split-K reduce is the same fold taken over the split index s.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_INDEX -2
#define OR_ERR_DUP_KEY -3
#define OR_ERR_NOMEM -4

#define OR_F32 0
#define OR_BF16 1

/* ------------------------------------------------------------------ */
/* binary32 <-> bf16                                                   */
/* ------------------------------------------------------------------ */

static uint32_t or_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float or_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 is the top half of a binary32 pattern, so widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return or_float((uint32_t)h << 16); }

/*
 * Round a binary32 value to bf16, to nearest, ties to even (IEEE 754
 * roundTiesToEven).  The kept part is the high 16 bits; the discarded part is
 * the low 16 bits.  Discarded > half: round the kept part up; == half: round
 * up only if the kept part is odd; < half: truncate.  Rounding up is +1 on the
 * kept pattern, which carries into the exponent and turns the largest finite
 * value into infinity, as the standard requires.  A NaN stays a NaN: its sign
 * and high payload bits are kept and the quiet bit is set, so truncating the
 * payload cannot turn it into an infinity.
 */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = or_bits(f);
    uint32_t kept = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)(kept | 0x0040u);
    if (rest > 0x8000u || (rest == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

void oracle_f32_to_bf16_array(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}

/* ------------------------------------------------------------------ */
/* the canonical fold (steps 3-5 above)                                */
/* ------------------------------------------------------------------ */

/* `level` must hold ceil(n/32) floats. */
static float or_canonical_sum_buf(const float* p, int64_t n, float* level)
{
    if (n == 0) return 0.0f;                       /* step 5 */
    int64_t nc = (n + 31) / 32;
    for (int64_t k = 0; k < nc; ++k) {             /* step 3 */
        int64_t lo = 32 * k;
        int64_t hi = lo + 32 < n ? lo + 32 : n;
        float acc = p[lo];
        for (int64_t j = lo + 1; j < hi; ++j) acc = acc + p[j];
        level[k] = acc;
    }
    int64_t len = nc;                              /* step 4 */
    while (len > 1) {
        int64_t next = (len + 1) / 2;
        for (int64_t k = 0; 2 * k + 1 < len; ++k)
            level[k] = level[2 * k] + level[2 * k + 1];
        if (len % 2 == 1)
            level[next - 1] = level[len - 1];      /* odd one carried up */
        len = next;
    }
    return level[0];
}

/* Canonical sum of n binary32 terms.  Returns 0 and sets *ok = 0 on OOM. */
float oracle_canonical_sum(const float* p, int64_t n, int32_t* ok)
{
    int64_t nc = (n + 31) / 32;
    float* level = (float*)malloc((size_t)(nc > 0 ? nc : 1) * sizeof(float));
    if (!level) { if (ok) *ok = 0; return 0.0f; }
    float r = or_canonical_sum_buf(p, n, level);
    free(level);
    if (ok) *ok = 1;
    return r;
}

/* ------------------------------------------------------------------ */
/* destination lists: stable counting sort by destination              */
/* ------------------------------------------------------------------ */

typedef struct { int64_t key; int64_t row; } or_keyed;

static int or_cmp_keyed(const void* a, const void* b)
{
    const or_keyed* x = (const or_keyed*)a;
    const or_keyed* y = (const or_keyed*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return x->row < y->row ? -1 : (x->row > y->row ? 1 : 0);
}

/*
 * row_ptr[M+1], perm[N]: perm[row_ptr[m] .. row_ptr[m+1]) lists the physical
 * rows i with idx[i] == m in ascending order key (src_id[i], or i when src_id
 * is NULL).  Order keys must be distinct within one destination, otherwise
 * the order is not defined and OR_ERR_DUP_KEY is returned.  idx outside
 * [0, M) gives OR_ERR_INDEX.  This is step 1 above; the MoE backward's sort by
 * (expert id, original token id) in Ch 09 section 3.2 is the same ordering.
 */
int oracle_build_lists(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M,
                       int64_t* row_ptr, int64_t* perm)
{
    if (N < 0 || M < 0 || (N > 0 && !idx) || !row_ptr || (N > 0 && !perm)) return OR_ERR_ARG;
    for (int64_t i = 0; i < N; ++i)
        if (idx[i] < 0 || (int64_t)idx[i] >= M) return OR_ERR_INDEX;
    for (int64_t m = 0; m <= M; ++m) row_ptr[m] = 0;
    for (int64_t i = 0; i < N; ++i) row_ptr[idx[i] + 1] += 1;      /* counts */
    for (int64_t m = 0; m < M; ++m) row_ptr[m + 1] += row_ptr[m];   /* prefix sums */
    int64_t* fill = (int64_t*)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
    if (!fill) return OR_ERR_NOMEM;
    for (int64_t m = 0; m < M; ++m) fill[m] = row_ptr[m];
    for (int64_t i = 0; i < N; ++i) perm[fill[idx[i]]++] = i;       /* stable placement */
    free(fill);
    if (!src_id) return OR_OK;
    int64_t maxlen = 0;
    for (int64_t m = 0; m < M; ++m)
        if (row_ptr[m + 1] - row_ptr[m] > maxlen) maxlen = row_ptr[m + 1] - row_ptr[m];
    or_keyed* tmp = (or_keyed*)malloc((size_t)(maxlen > 0 ? maxlen : 1) * sizeof(or_keyed));
    if (!tmp) return OR_ERR_NOMEM;
    int rc = OR_OK;
    for (int64_t m = 0; m < M && rc == OR_OK; ++m) {
        int64_t lo = row_ptr[m], n = row_ptr[m + 1] - lo;
        for (int64_t j = 0; j < n; ++j) { tmp[j].key = src_id[perm[lo + j]]; tmp[j].row = perm[lo + j]; }
        qsort(tmp, (size_t)n, sizeof(or_keyed), or_cmp_keyed);
        for (int64_t j = 0; j < n; ++j) {
            if (j > 0 && tmp[j].key == tmp[j - 1].key) { rc = OR_ERR_DUP_KEY; break; }
            perm[lo + j] = tmp[j].row;
        }
    }
    free(tmp);
    return rc;
}

/* ------------------------------------------------------------------ */
/* scatter-reduce (steps 1-6)                                          */
/* ------------------------------------------------------------------ */

static float or_load(const void* base, int32_t dtype, int64_t off)
{
    if (dtype == OR_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[off]);
    return ((const float*)base)[off];
}

static void or_store(void* base, int32_t dtype, int64_t off, float v)
{
    if (dtype == OR_BF16) ((uint16_t*)base)[off] = oracle_f32_to_bf16(v);
    else ((float*)base)[off] = v;
}

/*
 * out[m][h] = canonical sum over the terms of destination m.
 * Physical row r lives in shard q, the first q with r < shard_rows[0] + ... +
 * shard_rows[q]; within it at local row r - (rows of earlier shards), element
 * h at x_shards[q][local * ldx + h].  Sharding only says where bytes live: the
 * order key is global, so the result cannot depend on P (the EP-size
 * invariance of the interview notes' "why pay the overhead" section).
 */
static int or_scatter(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M,
                      const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                      int32_t x_dtype, int64_t ldx, int64_t H, const float* w,
                      void* out, int64_t ldo, int32_t out_dtype, int accumulate)
{
    if (N < 0 || M < 0 || H < 0 || P < 1 || ldx < H || ldo < H || (M > 0 && H > 0 && !out))
        return OR_ERR_ARG;
    if ((x_dtype != OR_F32 && x_dtype != OR_BF16) || (out_dtype != OR_F32 && out_dtype != OR_BF16))
        return OR_ERR_ARG;
    int64_t total = 0;
    for (int32_t q = 0; q < P; ++q) { if (shard_rows[q] < 0) return OR_ERR_ARG; total += shard_rows[q]; }
    if (total != N) return OR_ERR_ARG;

    int64_t* row_ptr = (int64_t*)malloc((size_t)(M + 1) * sizeof(int64_t));
    int64_t* perm = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    int32_t* shard_of = (int32_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int32_t));
    int64_t* local_of = (int64_t*)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!row_ptr || !perm || !shard_of || !local_of) {
        free(row_ptr); free(perm); free(shard_of); free(local_of); return OR_ERR_NOMEM;
    }
    int rc = oracle_build_lists(idx, src_id, N, M, row_ptr, perm);
    if (rc != OR_OK) { free(row_ptr); free(perm); free(shard_of); free(local_of); return rc; }
    {
        int64_t r = 0;
        for (int32_t q = 0; q < P; ++q)
            for (int64_t l = 0; l < shard_rows[q]; ++l, ++r) { shard_of[r] = q; local_of[r] = l; }
    }
    int64_t maxlen = 0;
    for (int64_t m = 0; m < M; ++m)
        if (row_ptr[m + 1] - row_ptr[m] > maxlen) maxlen = row_ptr[m + 1] - row_ptr[m];
    float* terms = (float*)malloc((size_t)(maxlen > 0 ? maxlen : 1) * sizeof(float));
    float* level = (float*)malloc((size_t)((maxlen + 31) / 32 > 0 ? (maxlen + 31) / 32 : 1) * sizeof(float));
    if (!terms || !level) rc = OR_ERR_NOMEM;
    for (int64_t m = 0; m < M && rc == OR_OK; ++m) {
        int64_t lo = row_ptr[m], n = row_ptr[m + 1] - lo;
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t j = 0; j < n; ++j) {                    /* step 2 */
                int64_t i = perm[lo + j];
                float xv = or_load(x_shards[shard_of[i]], x_dtype, local_of[i] * ldx + h);
                float p = w ? w[i] * xv : xv;
                terms[j] = p;
            }
            float sum = or_canonical_sum_buf(terms, n, level);
            if (accumulate) {
                if (n == 0) continue;                       /* untouched */
                sum = or_load(out, out_dtype, m * ldo + h) + sum;  /* one binary32 add */
            }
            or_store(out, out_dtype, m * ldo + h, sum);
        }
    }
    free(terms); free(level);
    free(row_ptr); free(perm); free(shard_of); free(local_of);
    return rc;
}

int oracle_scatter_reduce(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M,
                          const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                          int32_t x_dtype, int64_t ldx, int64_t H, const float* w,
                          void* out, int64_t ldo, int32_t out_dtype)
{
    return or_scatter(idx, src_id, N, M, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, 0);
}

/*
 * index_add_ semantics (Megatron-LM determinism developer reference, section
 * 3.1 op catalog: index_add_ is the deterministic replacement of the atomic
 * scatter_add_): each destination with at least one term becomes
 * out[m] + S[m], one binary32 add of the canonical sum S[m] to the value
 * already there, then stored as out_dtype; destinations without terms are
 * left as they are.
 */
int oracle_index_add(const int32_t* idx, const int64_t* src_id, int64_t N, int64_t M,
                     const void* const* x_shards, const int64_t* shard_rows, int32_t P,
                     int32_t x_dtype, int64_t ldx, int64_t H, const float* w,
                     void* out, int64_t ldo, int32_t out_dtype)
{
    return or_scatter(idx, src_id, N, M, x_shards, shard_rows, P, x_dtype, ldx, H, w, out, ldo, out_dtype, 1);
}

/*
 * Split-K reduce: out[e] = canonical sum of partials[s * ldp + e] over
 * s = 0 .. S-1 in split-id order, no multiply (Ch 09, section 3.3: each split
 * writes its own buffer and a reduce kernel sums them in split-id order).
 */
int oracle_splitk_reduce(const float* partials, int32_t S, int64_t count, int64_t ldp,
                         void* out, int32_t out_dtype)
{
    if (S < 0 || count < 0 || ldp < count || (count > 0 && !out) || (S > 0 && count > 0 && !partials))
        return OR_ERR_ARG;
    if (out_dtype != OR_F32 && out_dtype != OR_BF16) return OR_ERR_ARG;
    float* terms = (float*)malloc((size_t)(S > 0 ? S : 1) * sizeof(float));
    float* level = (float*)malloc((size_t)((S + 31) / 32 > 0 ? (S + 31) / 32 : 1) * sizeof(float));
    if (!terms || !level) { free(terms); free(level); return OR_ERR_NOMEM; }
    for (int64_t e = 0; e < count; ++e) {
        for (int32_t s = 0; s < S; ++s) terms[s] = partials[(int64_t)s * ldp + e];
        or_store(out, out_dtype, e, or_canonical_sum_buf(terms, S, level));
    }
    free(terms); free(level);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* fingerprint                                                         */
/* ------------------------------------------------------------------ */

/*
 * The repeatability gate compares a per-tensor fingerprint byte for byte
 * rather than a printed loss ("Bit-exact training interview notes", section
 * "how to verify: three gates").  The pages use torch.hash_tensor; this
 * library defines its own fingerprint so that any grid computes the same
 * value:
 *   words  = the buffer read as little-endian 64-bit words, the last one
 *            padded with zero bytes;
 *   h      = mix(nbytes ^ 0x6A09E667F3BCC909)
 *            + sum_j mix(word_j ^ (j * 0x9E3779B97F4A7C15))   (mod 2^64)
 * where mix is the SplitMix64 output finalizer (Steele, Lea, Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).  Addition mod
 * 2^64 is associative and commutative, so any summation order gives the same
 * u64.
 */
uint64_t oracle_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t oracle_hash(const void* p, uint64_t nbytes)
{
    const uint8_t* b = (const uint8_t*)p;
    uint64_t h = oracle_mix64(nbytes ^ 0x6A09E667F3BCC909ull);
    uint64_t nwords = (nbytes + 7u) / 8u;
    for (uint64_t j = 0; j < nwords; ++j) {
        uint64_t word = 0;
        for (uint64_t k = 0; k < 8u; ++k) {
            uint64_t at = 8u * j + k;
            uint64_t byte = at < nbytes ? (uint64_t)b[at] : 0u;
            word |= byte << (8u * k);
        }
        h += oracle_mix64(word ^ (j * 0x9E3779B97F4A7C15ull));
    }
    return h;
}

/* ------------------------------------------------------------------ */
/* sorted router top-k and the MoE dispatch layout                     */
/* ------------------------------------------------------------------ */

/*
 * The sorted router top-k is one of the hot spots of the deterministic path
 * ("Megatron-LM determinism developer reference", section 3.3); the pages
 * give no tie rule, so this library fixes one:
 *   - scores are ordered by IEEE 754 totalOrder (so -0.0 < +0.0, +inf below
 *     every positive NaN, -inf above every negative NaN): the unsigned order
 *     of the bit pattern with its sign bit set when it was clear, and all
 *     bits inverted when it was set;
 *   - among equal bit patterns the lower expert id ranks first.
 * Position r of token t's list is the r-th greatest score under that order.
 */
static uint32_t or_total_order_key(float f)
{
    uint32_t u = or_bits(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/*
 * ids[t][r], w[t][r] for r < k: the selection by repeated maximum -- round r
 * takes, among the experts not taken yet, the one of greatest key, scanning e
 * upwards and replacing only on a strictly greater key (so the lowest id
 * wins a tie).  renormalize != 0: sum = w[0] + w[1] + ... + w[k-1] added
 * left to right in binary32 from w[0], then each w[r] = fl32(w[r] / sum).
 * scores[t][e] sits at scores[t * lds + e].  1 <= k <= E.
 */
int oracle_router_topk(const float* scores, int64_t T, int32_t E, int64_t lds, int32_t k, int32_t renormalize,
                       int32_t* ids, float* w)
{
    if (T < 0 || E < 1 || k < 1 || k > E || lds < E || (T > 0 && (!scores || !ids || !w))) return OR_ERR_ARG;
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!taken) return OR_ERR_NOMEM;
    for (int64_t t = 0; t < T; ++t) {
        const float* s = scores + t * lds;
        memset(taken, 0, (size_t)E);
        for (int32_t r = 0; r < k; ++r) {
            int32_t best = -1;
            uint32_t best_key = 0;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                uint32_t key = or_total_order_key(s[e]);
                if (best < 0 || key > best_key) { best = e; best_key = key; }
            }
            taken[best] = 1;
            ids[t * k + r] = best;
            w[t * k + r] = s[best];
        }
        if (renormalize) {
            float sum = w[t * k];
            for (int32_t r = 1; r < k; ++r) sum = sum + w[t * k + r];
            for (int32_t r = 0; r < k; ++r) w[t * k + r] = w[t * k + r] / sum;
        }
    }
    free(taken);
    return OR_OK;
}

/*
 * The dispatch layout of top-k routing: slot i = t * k + j (token t's j-th
 * choice, expert ids[i]) goes to dispatch row slot_row[i], the rows grouped
 * by expert in ascending expert id and, inside an expert, in ascending slot
 * -- for distinct choices per token the stable (expert id, original token
 * id) order of the MoE backward ("DeepSeek-V4 book, Ch 09", section 3.2).
 * Written as the textbook stable counting sort:
 *   expert_offsets[e] = number of slots whose expert is below e (E+1 values);
 *   walking the slots upwards, each takes the next free row of its expert;
 *   row_token[p] = token of the slot at row p, row_w[p] = its weight (w may
 *   be NULL, then row_w is not written).
 * An expert id outside [0, E) gives OR_ERR_INDEX.
 */
int oracle_moe_route(const int32_t* ids, const float* w, int64_t T, int32_t k, int32_t E,
                     int64_t* expert_offsets, int32_t* row_token, float* row_w, int32_t* slot_row)
{
    if (T < 0 || k < 0 || E < 1 || !expert_offsets) return OR_ERR_ARG;
    const int64_t N = T * (int64_t)k;
    if (N > 0 && (!ids || !row_token || !slot_row || (w && !row_w))) return OR_ERR_ARG;
    for (int64_t i = 0; i < N; ++i)
        if (ids[i] < 0 || ids[i] >= E) return OR_ERR_INDEX;
    for (int32_t e = 0; e <= E; ++e) expert_offsets[e] = 0;
    for (int64_t i = 0; i < N; ++i) expert_offsets[ids[i] + 1] += 1;     /* counts */
    for (int32_t e = 0; e < E; ++e) expert_offsets[e + 1] += expert_offsets[e];
    int64_t* next = (int64_t*)malloc((size_t)E * sizeof(int64_t));
    if (!next) return OR_ERR_NOMEM;
    for (int32_t e = 0; e < E; ++e) next[e] = expert_offsets[e];
    for (int64_t i = 0; i < N; ++i) {
        int64_t p = next[ids[i]]++;
        slot_row[i] = (int32_t)p;
        row_token[p] = (int32_t)(i / k);
        if (w) row_w[p] = w[i];
    }
    free(next);
    return OR_OK;
}
