/* Oracle for the routed-expert MoE block -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, CPU implementation in double precision of what the block computes. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may call it; the product path
 * (the CUDA library) never does and shares no code with it.
 *
 * Sources (titles of the web pages that describe the Strata engine and its model):
 *   [satyajit] "Strata engine" code reading, ai.thesatyajit.com -- sections "The byte budget, in
 *              code" (dimensions, Q2_0 blob size) and "The CPU kernels" (Q2_0 code meaning and the
 *              in-block bit order of unpack64_q2_0).
 *   [zwxr]     zwxr.cn news/242664, section "一次路由的完整旅程" (one routing's full journey): router
 *              logits from a BF16 GEMV, softmax over all 512, stable descending argsort, top-10,
 *              renormalise with ggml's lower clamp, then the weighted combine of the parts.
 *   [momoyeyu] momoyeyu.github.io "ai-infra-strata", sections "搬权重与搬向量" (an expert maps x to
 *              y of the same width), "提示词处理" (tokens gathered per expert) and "权重映射"
 *              (gate, up and down stored together).
 *   [wayneh]   wayneh.tw "strata-local-moe-inference": 48 layers x 512 experts, top-10.
 * The SwiGLU form down(silu(gate x) * (up x)), the rmsnorm residual stack and the synthetic
 * inputs are the benchmark's statement of the block; the pages never print them.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - Q2_0 block = {fp16 d, 16 code bytes} (18 B; the blob size fixes 18), weight i of a block at
 *     code byte i/4, bits 2*(i%4); value d*(c - q2_offset); the pages say codes {0,1,2,3} mean
 *     {-1,0,1,2}*scale, i.e. q2_offset = 1; the benchmark text says c-2, so both are supported.
 *   - blocks are runs of 64 consecutive weights of the row-major matrix; gate and up are
 *     [FF rows][H cols] (x -> FF), down is [H rows][FF cols].
 *   - ggml's lower clamp on the renormalising sum: 2^-14 (never active for top-10 of 512).
 *   - stable descending order: equal probabilities keep the lower expert id first.
 *   - grouping: pairs (t, k) numbered p = t*K + k, sorted by expert, ascending p within an expert.
 *   - rmsnorm: x / sqrt(mean(x^2) + 1e-6), no gain.
 */
#ifndef STRATA_ORACLE_H
#define STRATA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double oracle_fp16_to_double(uint16_t h);
double oracle_bf16_to_double(uint16_t b);

/* 2-bit code of weight i (0..63) of a Q2_0 block's 16 code bytes. */
int oracle_q2_code(const uint8_t* codes16, int i);

/* Dequantise n_blocks consecutive canonical blocks into 64*n_blocks doubles. */
void oracle_dequant_blocks(const uint8_t* blocks, int64_t n_blocks, int q2_offset, double* w);

/* Whole blob -> dense gate[FF][H], up[FF][H], down[H][FF]. Returns 0, or -1 if H*FF % 64 != 0. */
int oracle_dequant_blob(const uint8_t* blob, int H, int FF, int q2_offset,
                        double* gate, double* up, double* down);

/* logits[e] = sum_h xn[h] * Wr[e][h] (+ bias[e]); Wr bf16 bit patterns [E][H]; bias may be NULL. */
void oracle_router_logits(const double* xn, int H, int E, const uint16_t* w_router,
                          const float* bias, double* logits);

/* Softmax over E, stable descending order, first K ids, renormalised weights (clamped sum).
 * p_out (nullable) receives the E probabilities. */
void oracle_top_k(const double* logits, int E, int K, int32_t* ids, double* w, double* p_out);

/* Weights for a given id set (teacher forcing): w_k = p[ids[k]] / max(sum_j p[ids[j]], 2^-14). */
void oracle_weights_for_ids(const double* logits, int E, int K, const int32_t* ids, double* w);

/* Counting sort of the T*K pairs by expert. expert_off[E+1], pair[T*K], active[E], n_active[1]. */
void oracle_group(const int32_t* ids, int T, int K, int E, int32_t* expert_off, int32_t* pair,
                  int32_t* active, int32_t* n_active);

/* One expert on one token: y = down(silu(gate x) * (up x)), straight from the canonical blob. */
void oracle_expert(const uint8_t* blob, int H, int FF, int q2_offset, const double* x, double* y);

/* x / sqrt(mean(x^2) + eps). */
void oracle_rmsnorm(const double* x, int H, double eps, double* xn);

/* Steps 1-2 only for T tokens (router input = x, or rmsnorm(x) when residual): ids [T][K],
 * w [T][K], logits [T][E] (each nullable). n_threads splits tokens. Returns 0 or -1. */
int oracle_route_tokens(const float* x, int T, int H, int E, int K, const uint16_t* w_router,
                        const float* bias, int residual, int32_t* ids_out, double* w_out,
                        double* logits_out, int n_threads);

/* One MoE layer for T tokens.
 *   x: fp32 [T][H].  w_router: bf16 [E][H].  bias: fp32 [E] or NULL.
 *   blobs: E pointers to canonical blobs (an entry may be NULL if that expert is never routed).
 *   residual = 0: out = moe(x);  residual = 1: out = x + moe(rmsnorm(x)) (router and experts
 *   both read rmsnorm(x)).
 *   ids_in (nullable) [T][K]: routing to use instead of the oracle's own top-K (teacher forcing);
 *   weights are then the oracle's probabilities renormalised over that id set.
 *   Outputs (each nullable except out): ids_out [T][K], w_out [T][K], logits_out [T][E],
 *   parts_out [T][K][H] (unweighted expert outputs), out [T][H].
 *   n_threads >= 1 splits tokens; results do not depend on it.
 *   shared_blob (nullable): the layer's shared expert (canonical blob of the routed experts' shape);
 *   its output on the same input is added with weight 1 after the routed combine, before the
 *   residual.  Reading: the pages name a shared expert run for every token but give neither its width
 *   nor a gate.
 * Returns 0, or -1 on a bad argument / a NULL blob that routing needs. */
int oracle_moe_layer(const float* x, int T, int H, int FF, int E, int K, const uint16_t* w_router,
                     const float* bias, const uint8_t* const* blobs, int q2_offset, int residual,
                     const int32_t* ids_in, int32_t* ids_out, double* w_out, double* logits_out,
                     double* parts_out, double* out, int n_threads, const uint8_t* shared_blob);

#ifdef __cplusplus
}
#endif
#endif
