/* Oracle for the routed-expert MoE block -- TEST INFRASTRUCTURE ONLY (see strata_oracle.h).
 * Plain loops in double precision; no blocking, no SIMD, no fused multiply-add contraction
 * (built with -ffp-contract=off so x86 and Arm hosts give the same bits). */
#include "strata_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* IEEE binary16 -> double, written out from the format's definition. */
double oracle_fp16_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exp = (h >> 10) & 0x1F;
  const int man = h & 0x3FF;
  double v;
  if (exp == 0) {
    v = ldexp((double)man, -24); /* subnormal: man * 2^-14 * 2^-10 */
  } else if (exp == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = ldexp((double)(man | 0x400), exp - 25); /* (1024 + man) * 2^(exp-15-10) */
  }
  return sign ? -v : v;
}

/* bf16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
  union {
    uint32_t u;
    float f;
  } c;
  c.u = (uint32_t)b << 16;
  return (double)c.f;
}

/* [satyajit] "The CPU kernels": 16 bytes hold 64 codes; unpack64_q2_0 widens them to 8 x u16 and
 * shifts each 16-bit lane by 0, 2, ..., 14, so weight i sits in byte i/4 at bits 2*(i%4). */
int oracle_q2_code(const uint8_t* codes16, int i) { return (codes16[i >> 2] >> (2 * (i & 3))) & 3; }

/* [satyajit] "The byte budget, in code": 64 weights = 16 bytes of 2-bit codes + an fp16 scale;
 * "The CPU kernels": codes {0,1,2,3} mean {-1,0,1,2} x scale, i.e. w = d * (c - q2_offset). */
void oracle_dequant_blocks(const uint8_t* blocks, int64_t n_blocks, int q2_offset, double* w) {
  for (int64_t b = 0; b < n_blocks; ++b) {
    const uint8_t* blk = blocks + 18 * b;
    const uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    const double d = oracle_fp16_to_double(dbits);
    for (int i = 0; i < 64; ++i) w[64 * b + i] = d * (double)(oracle_q2_code(blk + 2, i) - q2_offset);
  }
}

/* [momoyeyu] "权重映射": gate, up and down sit together; [satyajit]: each is 2,560 x 640 and the
 * blob is 3 * H*FF*18/64 bytes.  Order gate, up, down. */
int oracle_dequant_blob(const uint8_t* blob, int H, int FF, int q2_offset, double* gate, double* up,
                        double* down) {
  const int64_t n = (int64_t)H * FF;
  if (n % 64) return -1;
  const int64_t nb = n / 64;
  oracle_dequant_blocks(blob, nb, q2_offset, gate);
  oracle_dequant_blocks(blob + 18 * nb, nb, q2_offset, up);
  oracle_dequant_blocks(blob + 36 * nb, nb, q2_offset, down);
  return 0;
}

/* [zwxr] "一次路由的完整旅程": moe_route projects the normalised activation with a BF16 GEMV to
 * 512 expert logits.  The optional bias is the benchmark's per-expert Zipf prior. */
void oracle_router_logits(const double* xn, int H, int E, const uint16_t* w_router, const float* bias,
                          double* logits) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    const uint16_t* row = w_router + (int64_t)e * H;
    for (int h = 0; h < H; ++h) acc += oracle_bf16_to_double(row[h]) * xn[h];
    if (bias) acc += (double)bias[e];
    logits[e] = acc;
  }
}

static const double kRenormFloor = 6.103515625e-05; /* 2^-14 */

static void softmax(const double* logits, int E, double* p) {
  double m = logits[0];
  for (int e = 1; e < E; ++e)
    if (logits[e] > m) m = logits[e];
  double z = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = exp(logits[e] - m);
    z += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= z;
}

/* [zwxr] "一次路由的完整旅程": native_router_top10 takes a softmax over all 512 experts, a stable
 * descending argsort, gathers the first 10 and renormalises with ggml's lower clamp. The first K
 * entries of a stable descending sort are taken by repeated selection of the largest remaining
 * probability, the lower id winning ties. */
void oracle_top_k(const double* logits, int E, int K, int32_t* ids, double* w, double* p_out) {
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
  softmax(logits, E, p);
  double s = 0.0;
  for (int k = 0; k < K; ++k) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || p[e] > p[best]) best = e;
    }
    taken[best] = 1;
    ids[k] = best;
    s += p[best];
  }
  const double denom = s > kRenormFloor ? s : kRenormFloor;
  for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / denom;
  if (p_out) memcpy(p_out, p, sizeof(double) * (size_t)E);
  free(taken);
  free(p);
}

void oracle_weights_for_ids(const double* logits, int E, int K, const int32_t* ids, double* w) {
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  softmax(logits, E, p);
  double s = 0.0;
  for (int k = 0; k < K; ++k) s += p[ids[k]];
  const double denom = s > kRenormFloor ? s : kRenormFloor;
  for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / denom;
  free(p);
}

/* [momoyeyu] "提示词处理": tokens routed to the same expert are gathered so one read of its weights
 * serves all of them.  A counting sort of pair numbers p = t*K + k by expert id, ascending p within
 * an expert; active lists the experts with at least one pair, in increasing id. */
void oracle_group(const int32_t* ids, int T, int K, int E, int32_t* expert_off, int32_t* pair,
                  int32_t* active, int32_t* n_active) {
  int32_t* count = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int p = 0; p < T * K; ++p) count[ids[p]]++;
  expert_off[0] = 0;
  for (int e = 0; e < E; ++e) expert_off[e + 1] = expert_off[e] + count[e];
  int na = 0;
  for (int e = 0; e < E; ++e)
    if (count[e]) active[na++] = e;
  *n_active = na;
  memset(count, 0, sizeof(int32_t) * (size_t)E);
  for (int p = 0; p < T * K; ++p) {
    const int e = ids[p];
    pair[expert_off[e] + count[e]++] = p;
  }
  free(count);
}

/* Weight (row r, col c) of a row-major [rows][cols] Q2_0 matrix stored as canonical blocks. */
static double q2_weight(const uint8_t* mat, int cols, int r, int c, int q2_offset) {
  const int64_t flat = (int64_t)r * cols + c;
  const uint8_t* blk = mat + 18 * (flat / 64);
  const double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
  return d * (double)(oracle_q2_code(blk + 2, (int)(flat % 64)) - q2_offset);
}

/* [momoyeyu] "搬权重与搬向量": an expert maps x (H) to y (H).  Its form, from the benchmark's
 * statement: y = down(silu(gate x) * (up x)), silu(z) = z / (1 + e^-z); gate and up are FF x H,
 * down is H x FF. */
void oracle_expert(const uint8_t* blob, int H, int FF, int q2_offset, const double* x, double* y) {
  const int64_t nb = (int64_t)H * FF / 64;
  const uint8_t* gate = blob;
  const uint8_t* up = blob + 18 * nb;
  const uint8_t* down = blob + 36 * nb;
  double* hbuf = (double*)malloc(sizeof(double) * (size_t)FF);
  for (int r = 0; r < FF; ++r) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += q2_weight(gate, H, r, c, q2_offset) * x[c];
      u += q2_weight(up, H, r, c, q2_offset) * x[c];
    }
    hbuf[r] = g / (1.0 + exp(-g)) * u;
  }
  for (int n = 0; n < H; ++n) {
    double acc = 0.0;
    for (int r = 0; r < FF; ++r) acc += q2_weight(down, FF, n, r, q2_offset) * hbuf[r];
    y[n] = acc;
  }
  free(hbuf);
}

void oracle_rmsnorm(const double* x, int H, double eps, double* xn) {
  double ss = 0.0;
  for (int h = 0; h < H; ++h) ss += x[h] * x[h];
  const double inv = 1.0 / sqrt(ss / (double)H + eps);
  for (int h = 0; h < H; ++h) xn[h] = x[h] * inv;
}

typedef struct {
  const float* x;
  int T, H, FF, E, K;
  const uint16_t* w_router;
  const float* bias;
  const uint8_t* const* blobs;
  const uint8_t* shared_blob;
  int q2_offset, residual;
  const int32_t* ids_in;
  int32_t* ids_out;
  double* w_out;
  double* logits_out;
  double* parts_out;
  double* out;
  int n_threads, tid;
  int err;
} layer_job;

/* One token: [zwxr] route -> top-10 -> experts -> "Combine" out = sum_k w_k * parts_k (k order),
 * then, when the layer has one, the shared expert's output on the same normalised input added with
 * weight 1 ([wayneh] lists a shared expert that runs for every token; its size and any gate are not on
 * the pages: it is read as an expert of the routed experts' shape and format, ungated), then the
 * residual for stacked layers. */
static int token_forward(const layer_job* j, int t) {
  const int H = j->H, E = j->E, K = j->K;
  double* xin = (double*)malloc(sizeof(double) * (size_t)H);
  double* xn = (double*)malloc(sizeof(double) * (size_t)H);
  double* logits = (double*)malloc(sizeof(double) * (size_t)E);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  double* w = (double*)malloc(sizeof(double) * (size_t)K);
  double* acc = j->out + (int64_t)t * H;
  int rc = 0;
  for (int h = 0; h < H; ++h) xin[h] = (double)j->x[(int64_t)t * H + h];
  if (j->residual)
    oracle_rmsnorm(xin, H, 1e-6, xn);
  else
    memcpy(xn, xin, sizeof(double) * (size_t)H);
  oracle_router_logits(xn, H, E, j->w_router, j->bias, logits);
  if (j->ids_in) {
    memcpy(ids, j->ids_in + (int64_t)t * K, sizeof(int32_t) * (size_t)K);
    for (int k = 0; k < K; ++k)
      if (ids[k] < 0 || ids[k] >= E) rc = -1;
    if (!rc) oracle_weights_for_ids(logits, E, K, ids, w);
  } else {
    oracle_top_k(logits, E, K, ids, w, NULL);
  }
  if (!rc) {
    for (int h = 0; h < H; ++h) acc[h] = 0.0;
    for (int k = 0; k < K; ++k) {
      const uint8_t* blob = j->blobs[ids[k]];
      if (!blob) {
        rc = -1;
        break;
      }
      oracle_expert(blob, H, j->FF, j->q2_offset, xn, y);
      if (j->parts_out) memcpy(j->parts_out + ((int64_t)t * K + k) * H, y, sizeof(double) * (size_t)H);
      for (int h = 0; h < H; ++h) acc[h] += w[k] * y[h];
    }
    if (!rc && j->shared_blob) {
      oracle_expert(j->shared_blob, H, j->FF, j->q2_offset, xn, y);
      for (int h = 0; h < H; ++h) acc[h] += y[h];
    }
    if (!rc && j->residual)
      for (int h = 0; h < H; ++h) acc[h] = xin[h] + acc[h];
  }
  if (j->ids_out) memcpy(j->ids_out + (int64_t)t * K, ids, sizeof(int32_t) * (size_t)K);
  if (j->w_out) memcpy(j->w_out + (int64_t)t * K, w, sizeof(double) * (size_t)K);
  if (j->logits_out) memcpy(j->logits_out + (int64_t)t * E, logits, sizeof(double) * (size_t)E);
  free(xin);
  free(xn);
  free(logits);
  free(y);
  free(ids);
  free(w);
  return rc;
}

static void* layer_worker(void* arg) {
  layer_job* j = (layer_job*)arg;
  for (int t = j->tid; t < j->T; t += j->n_threads)
    if (token_forward(j, t)) j->err = -1;
  return NULL;
}

int oracle_moe_layer(const float* x, int T, int H, int FF, int E, int K, const uint16_t* w_router,
                     const float* bias, const uint8_t* const* blobs, int q2_offset, int residual,
                     const int32_t* ids_in, int32_t* ids_out, double* w_out, double* logits_out,
                     double* parts_out, double* out, int n_threads, const uint8_t* shared_blob) {
  if (T < 0 || H <= 0 || FF <= 0 || E <= 0 || K <= 0 || K > E || !out || !x || !w_router || !blobs)
    return -1;
  if (((int64_t)H * FF) % 64) return -1;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > T) n_threads = T > 0 ? T : 1;
  layer_job* jobs = (layer_job*)calloc((size_t)n_threads, sizeof(layer_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  for (int i = 0; i < n_threads; ++i) {
    layer_job* j = &jobs[i];
    j->x = x;
    j->T = T;
    j->H = H;
    j->FF = FF;
    j->E = E;
    j->K = K;
    j->w_router = w_router;
    j->bias = bias;
    j->blobs = blobs;
    j->shared_blob = shared_blob;
    j->q2_offset = q2_offset;
    j->residual = residual;
    j->ids_in = ids_in;
    j->ids_out = ids_out;
    j->w_out = w_out;
    j->logits_out = logits_out;
    j->parts_out = parts_out;
    j->out = out;
    j->n_threads = n_threads;
    j->tid = i;
  }
  int rc = 0;
  if (n_threads == 1) {
    layer_worker(&jobs[0]);
  } else {
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, layer_worker, &jobs[i]);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  }
  for (int i = 0; i < n_threads; ++i)
    if (jobs[i].err) rc = -1;
  free(jobs);
  free(th);
  return rc;
}

typedef struct {
  const float* x;
  int T, H, E, K;
  const uint16_t* w_router;
  const float* bias;
  int residual;
  int32_t* ids_out;
  double* w_out;
  double* logits_out;
  int n_threads, tid;
} route_job;

static void* route_worker(void* arg) {
  route_job* j = (route_job*)arg;
  double* xn = (double*)malloc(sizeof(double) * (size_t)j->H);
  double* logits = (double*)malloc(sizeof(double) * (size_t)j->E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)j->K);
  double* w = (double*)malloc(sizeof(double) * (size_t)j->K);
  for (int t = j->tid; t < j->T; t += j->n_threads) {
    for (int h = 0; h < j->H; ++h) xn[h] = (double)j->x[(int64_t)t * j->H + h];
    if (j->residual) oracle_rmsnorm(xn, j->H, 1e-6, xn);
    oracle_router_logits(xn, j->H, j->E, j->w_router, j->bias, logits);
    oracle_top_k(logits, j->E, j->K, ids, w, NULL);
    if (j->ids_out) memcpy(j->ids_out + (int64_t)t * j->K, ids, sizeof(int32_t) * (size_t)j->K);
    if (j->w_out) memcpy(j->w_out + (int64_t)t * j->K, w, sizeof(double) * (size_t)j->K);
    if (j->logits_out) memcpy(j->logits_out + (int64_t)t * j->E, logits, sizeof(double) * (size_t)j->E);
  }
  free(xn);
  free(logits);
  free(ids);
  free(w);
  return NULL;
}

int oracle_route_tokens(const float* x, int T, int H, int E, int K, const uint16_t* w_router,
                        const float* bias, int residual, int32_t* ids_out, double* w_out,
                        double* logits_out, int n_threads) {
  if (T < 0 || H <= 0 || E <= 0 || K <= 0 || K > E || !x || !w_router) return -1;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > T) n_threads = T > 0 ? T : 1;
  route_job* jobs = (route_job*)calloc((size_t)n_threads, sizeof(route_job));
  pthread_t* th = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
  for (int i = 0; i < n_threads; ++i) {
    route_job* j = &jobs[i];
    j->x = x;
    j->T = T;
    j->H = H;
    j->E = E;
    j->K = K;
    j->w_router = w_router;
    j->bias = bias;
    j->residual = residual;
    j->ids_out = ids_out;
    j->w_out = w_out;
    j->logits_out = logits_out;
    j->n_threads = n_threads;
    j->tid = i;
  }
  if (n_threads == 1) {
    route_worker(&jobs[0]);
  } else {
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, route_worker, &jobs[i]);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  }
  free(jobs);
  free(th);
  return 0;
}
