/*
 * CPU oracle for the two steps that prepare an MLA decode call.  TEST
 * INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg call
 * it; the library never does.  It shares no code with the CUDA path.
 *
 * The pages name the decode kernel these steps feed (the TileLang talk,
 * "Tile级原语与自动推理机制融合，TileAI社区发起人深度剖析TileLang核心技术与优势",
 * section 什么是「TileLang」: the DeepSeek MLA kernel) but say nothing of how
 * its inputs are made.  The reading taken is DeepSeek's MLA decode step:
 *
 * 1. Cache append.  The s_q new tokens of batch entry b are the last s_q
 *    positions of its sequence, t = L_b - s_q + i for i < s_q, where L_b =
 *    cache_seqlens[b] already counts them (the convention of the decode
 *    call).  Token t's 576-wide row (512 latent + 64 rotary dims, bf16) goes
 *    to kv_cache[block_table[b][t / 64]][t % 64][0][0:576], bit for bit.
 *    Nothing else in the cache changes.
 *
 * 2. Query absorption.  With the key up-projection W_UK folded into the
 *    query, the decode query of head h is
 *        q_latent[b][i][h][c] = sum_{d < d_nope} q_nope[b][i][h][d] * W_UK[h][d][c]
 *    for c < d_c (d_nope = 128, d_c = 512 in DeepSeek's MLA), evaluated in
 *    fp64 from the bf16 inputs; the decode kernel's query row is
 *    [q_latent | q_rope].
 *
 * Every sum is a plain loop in the order written; there is no blocking or
 * reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ROW 576
#define PAGE 64

static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* 1. Returns 0, or -1 (and writes nothing at all) when a new token's
 * position or page is out of range. */
int oracle_cache_append(const uint16_t* kv_new, uint16_t* kv_cache, int num_pages,
                        const int32_t* block_table, int max_pages, const int32_t* seqlens,
                        int batch, int s_q)
{
    for (int pass = 0; pass < 2; ++pass) {
        for (int b = 0; b < batch; ++b) {
            for (int i = 0; i < s_q; ++i) {
                const int t = seqlens[b] - s_q + i;
                if (t < 0 || t / PAGE >= max_pages)
                    return -1;
                const int page = block_table[(size_t)b * max_pages + t / PAGE];
                if (page < 0 || page >= num_pages)
                    return -1;
                if (pass == 1) {
                    const uint16_t* src = kv_new + ((size_t)b * s_q + i) * ROW;
                    uint16_t* dst = kv_cache + ((size_t)page * PAGE + t % PAGE) * ROW;
                    for (int d = 0; d < ROW; ++d)
                        dst[d] = src[d];
                }
            }
        }
    }
    return 0;
}

/* 2. q_nope [rows][h_q][d_nope] bf16, w_uk [h_q][d_nope][d_c] bf16 ->
 * out [rows][h_q][d_c] fp64, rows = batch * s_q. */
void oracle_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, int rows, int h_q, int d_nope,
                     int d_c, double* out)
{
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < h_q; ++h) {
            const uint16_t* q = q_nope + ((size_t)r * h_q + h) * d_nope;
            const uint16_t* w = w_uk + (size_t)h * d_nope * d_c;
            double* o = out + ((size_t)r * h_q + h) * d_c;
            for (int c = 0; c < d_c; ++c) {
                double acc = 0.0;
                for (int d = 0; d < d_nope; ++d)
                    acc += bf16_value(q[d]) * bf16_value(w[(size_t)d * d_c + c]);
                o[c] = acc;
            }
        }
    }
}

