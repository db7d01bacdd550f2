/*
 * attn_oracle.c -- the correctness oracle for paged, block-sparse batched
 * attention.  TEST INFRASTRUCTURE ONLY: nothing in the product library links,
 * loads or calls this file; only the tests, the smoke check and the bench's
 * CPU-baseline leg do.
 *
 * It is the plain definition of the result, written out in fp64, with no
 * blocking, no splitting and no online softmax:
 *
 *   FlashInfer (paper summary page), section "연구 방법론 / 1. 통합된 KV 캐시
 *   추상화": every KV storage (paged, radix tree, contiguous) is one
 *   block-sparse matrix whose column blocks are KV pages.  Here the blocks of
 *   request b are the pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]); the
 *   last one holds last_page_len[b] valid slots.
 *
 *   FlashInfer 0.6 wiki page, section "배경: LLM 디코드의 병목 구조": decode
 *   reads the keys and values of every cached token and takes the scaled dot
 *   product of the query with them, i.e. softmax(q K^T * scale) V.
 *
 *   FlashInfer 0.6 wiki page, section "커널 유형별 역할 / Decode 어텐션": GQA
 *   and MQA; query head h reads KV head h / (Hq/Hkv) (contiguous groups; the
 *   pages do not fix the mapping, this is the plain reading).
 *
 *   BatchAttention PR page, section "코드 분석 §1" (MaskMode template
 *   parameter): the causal mask is aligned to the bottom right, so query
 *   token t of a request with Lq queries and Lkv keys sees key j iff
 *   j <= Lkv - Lq + t.
 *
 * Mask and logit variants (FlashInfer 0.6 wiki page, section "Blackwell
 * (SM100/SM103) 전용 경로 / CuTe-DSL GQA Decode 커널": sliding-window and
 * attention-sink masking; FlashInfer paper summary, section "2. 유연한 어텐션
 * 변형 지원": user-defined logits transforms and masks).  The pages name the
 * variants without formulas; the plain readings used here:
 *   sliding window (window_left W >= 0, off when < 0): query token t, at
 *     position q_pos = Lkv - Lq + t (the bottom-right alignment of the causal
 *     mask), also needs j >= q_pos - W;
 *   attention sink (sink_tokens S >= 0): keys j < S stay visible whatever the
 *     window says (the causal bound still applies);
 *   logits soft-cap (cap > 0, off when 0): the logit fed to the softmax is
 *     cap * tanh(scale * q.k / cap) instead of scale * q.k.
 *
 * RoPE fused into attention (FlashInfer paper summary, section "주요 성능
 * 테스트 결과 / 2. 커널 수준 성능": a kernel fusing RoPE with attention; the
 * page gives no formula).
 * The plain reading, Llama style: before the dot product, q and every key are
 * rotated by their positions; dims i and i + d/2 form a pair rotated by
 * a = (pos / rope_scale) * rope_theta^(-2i/d):
 *   x_i' = x_i cos a - x_{i+d/2} sin a,   x_{i+d/2}' = x_{i+d/2} cos a + x_i sin a.
 * Key j sits at position j and query token t at Lkv - Lq + t (the alignment
 * of the causal mask).  The cache holds unrotated keys.
 *
 * LSE is the natural log of the sum of exp of the logits (the *scaled*, and
 * when capped the capped, scores).  A row that sees no key gets O = 0 and
 * LSE = -inf (the pages are silent; this is the identity of the merge
 * operator below).
 *
 * Merge of two partial states (the "process the dense and the sparse part
 * separately, then combine" of the paper summary's section 1, and the
 * split-KV of the wiki's SM103 MLA section):
 *   s = log(exp(s_a) + exp(s_b)),  o = exp(s_a - s) o_a + exp(s_b - s) o_b.
 *
 * Storage element types: IEEE binary16 and bfloat16 are decoded from their bit
 * definitions here (sign, exponent, fraction), exactly, into double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_FP16 = 0, ORC_BF16 = 1, ORC_FP32 = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_decode_fp16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_decode_bf16(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float x;
    memcpy(&x, &bits, sizeof x);
    return (double)x;
}

static double load_elem(const void* base, int dtype, int64_t idx)
{
    if (dtype == ORC_FP16) return orc_decode_fp16(((const uint16_t*)base)[idx]);
    if (dtype == ORC_BF16) return orc_decode_bf16(((const uint16_t*)base)[idx]);
    return (double)((const float*)base)[idx];
}

/* Everything that describes one batch of paged attention. */
typedef struct {
    int32_t batch;
    const int32_t* qo_indptr;     /* [batch+1] query tokens of request b: [qo_indptr[b], qo_indptr[b+1]) */
    const int32_t* kv_indptr;     /* [batch+1] pages of request b in kv_indices */
    const int32_t* kv_indices;    /* physical page ids */
    const int32_t* last_page_len; /* [batch] valid slots in the last page, 1..page_size */
    int32_t num_qo_heads, num_kv_heads, head_dim, page_size, causal;
    double sm_scale;
    int32_t dtype;                /* element type of q, k, v */
    const void* q;                /* [tokens, Hq, d] */
    int64_t q_stride_tok, q_stride_head;
    const void* k;                /* [pages, page_size, Hkv, d] */
    int64_t k_stride_page, k_stride_slot, k_stride_head;
    const void* v;
    int64_t v_stride_page, v_stride_slot, v_stride_head;
    int32_t window_left;          /* < 0: no sliding window */
    int32_t sink_tokens;          /* keys j < sink_tokens ignore the window */
    double logits_soft_cap;       /* 0: plain scaled logits */
    int32_t rope;                 /* 1: rotate q and k by position (RoPE) */
    double rope_theta, rope_scale;
} orc_problem;

/* RoPE rotation of x[0..d) at position pos, in place (pairs i, i + d/2). */
static void rope_rotate(const orc_problem* p, double* x, int64_t pos)
{
    const int half = p->head_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double a = ((double)pos / p->rope_scale) * pow(p->rope_theta, -2.0 * i / p->head_dim);
        const double c = cos(a), sn = sin(a);
        const double x0 = x[i], x1 = x[i + half];
        x[i] = x0 * c - x1 * sn;
        x[i + half] = x1 * c + x0 * sn;
    }
}

static int32_t kv_len_of(const orc_problem* p, int b)
{
    int32_t np = p->kv_indptr[b + 1] - p->kv_indptr[b];
    return np == 0 ? 0 : (np - 1) * p->page_size + p->last_page_len[b];
}

/* One query row: request b, query token t of that request, query head h.
 * Writes o[head_dim] and *lse.  scores is caller scratch of >= kv_len entries. */
static void attend_one(const orc_problem* p, int b, int t, int h, double* scores, double* o, double* lse)
{
    const int d = p->head_dim;
    const int group = p->num_qo_heads / p->num_kv_heads;
    const int hk = h / group;
    const int32_t lq = p->qo_indptr[b + 1] - p->qo_indptr[b];
    const int32_t lkv = kv_len_of(p, b);
    const int64_t row = (int64_t)p->qo_indptr[b] + t;

    /* keys j = 0 .. nvis-1 pass the length and causal bounds; of those, a
     * sliding window keeps j >= q_pos - W, and the sink keeps j < S anyway */
    const int64_t q_pos = (int64_t)lkv - lq + t; /* bottom-right aligned */
    int64_t nvis = lkv;
    if (p->causal && q_pos + 1 < nvis) nvis = q_pos + 1;
    if (nvis < 0) nvis = 0;
    const int64_t win_lo = p->window_left >= 0 ? q_pos - p->window_left : INT64_MIN;
    int64_t nseen = 0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;

    const int64_t qbase = row * p->q_stride_tok + (int64_t)h * p->q_stride_head;
    double qr[512], kr[512]; /* rotated q and key (RoPE only; head_dim <= 512) */
    if (p->rope) {
        for (int c = 0; c < d; ++c) qr[c] = load_elem(p->q, p->dtype, qbase + c);
        rope_rotate(p, qr, q_pos);
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        if (j < win_lo && j >= p->sink_tokens) {
            scores[j] = -INFINITY; /* outside the window and not a sink key */
            continue;
        }
        ++nseen;
        int64_t page = p->kv_indices[p->kv_indptr[b] + j / p->page_size];
        int64_t slot = j % p->page_size;
        int64_t kbase = page * p->k_stride_page + slot * p->k_stride_slot + (int64_t)hk * p->k_stride_head;
        double dot = 0.0;
        if (p->rope) {
            for (int c = 0; c < d; ++c) kr[c] = load_elem(p->k, p->dtype, kbase + c);
            rope_rotate(p, kr, j);
            for (int c = 0; c < d; ++c) dot += qr[c] * kr[c];
        } else {
            for (int c = 0; c < d; ++c)
                dot += load_elem(p->q, p->dtype, qbase + c) * load_elem(p->k, p->dtype, kbase + c);
        }
        double logit = p->sm_scale * dot;
        if (p->logits_soft_cap > 0.0) logit = p->logits_soft_cap * tanh(logit / p->logits_soft_cap);
        scores[j] = logit;
        if (scores[j] > m) m = scores[j];
    }
    if (nseen == 0) {
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        if (scores[j] != -INFINITY) sum += exp(scores[j] - m);
    const double l = m + log(sum);
    for (int64_t j = 0; j < nvis; ++j) {
        if (scores[j] == -INFINITY) continue;
        int64_t page = p->kv_indices[p->kv_indptr[b] + j / p->page_size];
        int64_t slot = j % p->page_size;
        int64_t vbase = page * p->v_stride_page + slot * p->v_stride_slot + (int64_t)hk * p->v_stride_head;
        double w = exp(scores[j] - l);
        for (int c = 0; c < d; ++c) o[c] += w * load_elem(p->v, p->dtype, vbase + c);
    }
    *lse = l;
}

static int32_t request_of_row(const orc_problem* p, int32_t row)
{
    for (int b = 0; b < p->batch; ++b)
        if (row >= p->qo_indptr[b] && row < p->qo_indptr[b + 1]) return b;
    return -1;
}

static int32_t max_kv_len(const orc_problem* p)
{
    int32_t mx = 1;
    for (int b = 0; b < p->batch; ++b) {
        int32_t l = kv_len_of(p, b);
        if (l > mx) mx = l;
    }
    return mx;
}

/* All rows: o[row][h][d], lse[row][h] for row in [0, qo_indptr[batch]).
 * Returns 0, or -1 when scratch could not be allocated. */
int orc_attention_all(const orc_problem* p, double* o, double* lse)
{
    const int64_t rows = p->qo_indptr[p->batch];
    const int64_t n = rows * p->num_qo_heads;
    const int32_t mx = max_kv_len(p);
    int failed = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)mx);
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < n; ++i) {
            if (!scores) continue;
            int32_t row = (int32_t)(i / p->num_qo_heads);
            int h = (int)(i % p->num_qo_heads);
            int b = request_of_row(p, row);
            attend_one(p, b, row - p->qo_indptr[b], h, scores, o + i * p->head_dim, lse + i);
        }
        free(scores);
    }
    return failed ? -1 : 0;
}

/* Selected (row, head) pairs only: o[i][d], lse[i].  Returns 0, -1 on
 * allocation failure, -2 when a row lies outside every request. */
int orc_attention_select(const orc_problem* p, int64_t n_sel, const int32_t* sel_row,
                         const int32_t* sel_head, double* o, double* lse)
{
    const int32_t mx = max_kv_len(p);
    int failed = 0;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)mx);
        if (!scores) {
#pragma omp atomic write
            failed = -1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_sel; ++i) {
            if (!scores) continue;
            int b = request_of_row(p, sel_row[i]);
            if (b < 0) {
#pragma omp atomic write
                failed = -2;
                continue;
            }
            attend_one(p, b, sel_row[i] - p->qo_indptr[b], sel_head[i], scores, o + i * p->head_dim, lse + i);
        }
        free(scores);
    }
    return failed;
}

/* Merge n pairs of states (o_a, s_a), (o_b, s_b) of width d each. */
void orc_merge_states(int64_t n, int32_t d, const double* o_a, const double* s_a, const double* o_b,
                      const double* s_b, double* o_out, double* s_out)
{
    for (int64_t i = 0; i < n; ++i) {
        double sa = s_a[i], sb = s_b[i];
        if (sa == -INFINITY && sb == -INFINITY) {
            for (int c = 0; c < d; ++c) o_out[i * d + c] = 0.0;
            s_out[i] = -INFINITY;
            continue;
        }
        double mx = sa > sb ? sa : sb;
        double s = mx + log(exp(sa - mx) + exp(sb - mx));
        double wa = exp(sa - s), wb = exp(sb - s);
        for (int c = 0; c < d; ++c) o_out[i * d + c] = wa * o_a[i * d + c] + wb * o_b[i * d + c];
        s_out[i] = s;
    }
}
