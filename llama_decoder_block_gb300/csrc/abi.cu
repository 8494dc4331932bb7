// C entry points: argument validation, workspace carve-up and the order of the steps
// of the pre-norm decoder layer ("05 LLaMA3 Block — 从零件到发动机" §4.2: save residual,
// norm, sublayer, add back -- twice) on top of the kernels of the other files.
#include <algorithm>
#include <cstring>
#include <utility>

#include "common.cuh"
#include "internal.h"

using namespace llama;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Carves consecutive aligned regions out of the caller's workspace.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  }
};

size_t esize(int dtype) { return dtype == LLAMA_BF16 ? 2 : 4; }

int check_dims(const llama_layer_dims* d) {
  if (d == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (d->d_model <= 0 || d->n_heads <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->d_inter <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (d->n_heads % d->n_kv_heads != 0) return LLAMA_ERR_INVALID_ARG;   // each KV head serves H/G query heads
  if (d->head_dim % 2 != 0) return LLAMA_ERR_INVALID_ARG;              // RoPE rotates pairs
  if (!(d->rms_eps >= 0.f)) return LLAMA_ERR_INVALID_ARG;
  if (d->dtype != LLAMA_F32 && d->dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (d->rope_style != LLAMA_ROPE_EVEN_ODD && d->rope_style != LLAMA_ROPE_HALF) return LLAMA_ERR_INVALID_ARG;
  if (d->dtype == LLAMA_BF16) {
    // the tensor-core path: 128-wide head tiles and 128-row weight blocks; decode attention
    // takes query heads in groups of up to 8 per KV head
    const int rep = d->n_heads / d->n_kv_heads;
    if (d->head_dim != 128 || d->d_model % 128 != 0 || d->d_inter % 128 != 0) return LLAMA_ERR_UNSUPPORTED;
    if (rep != 1 && rep != 2 && rep != 4 && rep % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  } else {
    if (d->head_dim > 256) return LLAMA_ERR_UNSUPPORTED;
  }
  return LLAMA_OK;
}

int check_weights(const llama_layer_weights* w) {
  if (w == nullptr) return LLAMA_ERR_INVALID_ARG;
  const void* ptrs[] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm, w->w_gate, w->w_up, w->w_down};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return LLAMA_ERR_INVALID_ARG;
  return LLAMA_OK;
}

struct PrefillWs {
  void *xn, *q, *o, *h, *a;
  int* sync;   // bf16: the grid-wide counts of the two GEMM prologues that normalise x and h
};

size_t prefill_ws(const llama_layer_dims* d, int B, int S, void* base, PrefillWs* out) {
  const size_t es = esize(d->dtype);
  const size_t M = static_cast<size_t>(B) * S;
  Carver c(base);
  PrefillWs w;
  w.xn = c.take(M * d->d_model * es);                      // RMSNorm output (both norms)
  w.q = c.take(M * d->n_heads * d->head_dim * es);         // [B, H, S, D]
  w.o = c.take(M * d->n_heads * d->head_dim * es);         // attention output [B, S, H*D]
  w.h = c.take(M * d->d_model * es);                       // attention half output
  w.a = c.take(M * d->d_inter * es);                       // SiLU(gate) * up
  w.sync = static_cast<int*>(c.take(d->dtype == LLAMA_BF16 ? 2 * sizeof(int) : 0));
  if (out) *out = w;
  return c.off;
}

struct DecodeWs {
  void *xn, *q, *o, *h, *a, *part, *attn;
};

size_t decode_part_floats(const llama_layer_dims* d, int B, int num_sms) {
  const int qkv = (d->n_heads + 2 * d->n_kv_heads) * d->head_dim;
  const int Ns[4] = {qkv, d->d_model, 2 * d->d_inter, d->d_model};
  const int Ks[4] = {d->d_model, d->n_heads * d->head_dim, d->d_model, d->d_inter};
  size_t mx = 0;
  for (int i = 0; i < 4; ++i) {
    const size_t s = static_cast<size_t>(choose_splits(num_sms, Ns[i], Ks[i], B));
    mx = std::max(mx, s * B * Ns[i]);
  }
  return mx;
}

size_t decode_ws(const llama_layer_dims* d, int B, int max_T, int num_sms, void* base, DecodeWs* out) {
  const size_t es = esize(d->dtype);
  Carver c(base);
  DecodeWs w;
  w.xn = c.take(static_cast<size_t>(B) * d->d_model * es);
  w.q = c.take(static_cast<size_t>(B) * d->n_heads * d->head_dim * es);
  w.o = c.take(static_cast<size_t>(B) * d->n_heads * d->head_dim * es);
  w.h = c.take(static_cast<size_t>(B) * d->d_model * es);
  w.a = c.take(static_cast<size_t>(B) * d->d_inter * es);
  if (d->dtype == LLAMA_BF16) {
    w.part = c.take(decode_part_floats(d, B, num_sms) * sizeof(float));
    w.attn = c.take(attn_decode_ws_bytes(B, d->n_heads, d->n_kv_heads, d->head_dim));
  } else {
    w.part = w.attn = nullptr;
  }
  if (out) *out = w;
  return c.off;
}

int num_sms_current(int* sms) {
  Ctx c;
  int rc = make_ctx(nullptr, &c);
  if (rc != LLAMA_OK) return rc;
  *sms = c.num_sms;
  return LLAMA_OK;
}

// start, lens: null (a prompt from position 0) or device [B] (a chunk on top of the cache).
// `c0` launches the first kernel (without programmatic serialisation when the call starts
// a new stream of work), `c` the others.  bf16 layers: `sync` (2 ints, zero) are the counts of
// the two GEMM prologues; null: the workspace's own, zeroed here.
int prefill_impl(const Ctx& c0, const Ctx& c_rest, const llama_layer_dims* d, const llama_layer_weights* w,
                 const void* x, void* out, const float* cos, const float* sin, int max_pos, llama_kv_cache cache,
                 int B, int S, void* ws, const int32_t* start = nullptr, const int32_t* lens = nullptr,
                 int* sync = nullptr) {
  PrefillWs p;
  prefill_ws(d, B, S, ws, &p);
  const Ctx& c = c_rest;
  const int M = B * S, dm = d->d_model, H = d->n_heads, G = d->n_kv_heads, D = d->head_dim, I = d->d_inter;
  int rc;
  if (d->dtype == LLAMA_BF16) {
    // Both RMSNorms run in the prologue of the GEMM that consumes them (the QKV and the gate/up
    // projections), which normalises the rows into xn and then streams them as its A operand.
    if (sync == nullptr) {
      sync = p.sync;
      if (cudaMemsetAsync(sync, 0, 2 * sizeof(int), c0.stream) != cudaSuccess) return LLAMA_ERR_CUDA;
    }
    const NormPro n1{w->attn_norm, d->rms_eps, p.xn, sync};
    const NormPro n2{w->ffn_norm, d->rms_eps, p.xn, sync + 1};
    if ((rc = gemm_qkv_rope(c0, x, w->wq, w->wk, w->wv, B, S, dm, H, G, D, cos, sin, p.q, cache.k, cache.v,
                            cache.max_T, d->rope_style, start, lens, max_pos, &n1)))
      return rc;
    if ((rc = attn_prefill_tc(c, p.q, cache.k, cache.v, p.o, B, S, H, G, D, cache.max_T, start, lens, max_pos)))
      return rc;
    if ((rc = gemm_residual(c, p.o, w->wo, x, p.h, M, dm, H * D))) return rc;
    if ((rc = gemm_swiglu(c, p.h, w->w_gate, w->w_up, p.a, M, I, dm, &n2))) return rc;
    return gemm_residual(c, p.a, w->w_down, p.h, out, M, dm, I);
  }
  if ((rc = rmsnorm(c0, x, w->attn_norm, p.xn, M, dm, d->rms_eps, d->dtype))) return rc;
  const float* xf = static_cast<const float*>(x);
  float* xn = static_cast<float*>(p.xn);
  float* h = static_cast<float*>(p.h);
  float* a = static_cast<float*>(p.a);
  if ((rc = simt_qkv_rope(c, xn, static_cast<const float*>(w->wq), static_cast<const float*>(w->wk),
                          static_cast<const float*>(w->wv), B, S, dm, H, G, D, cos, sin, start, max_pos,
                          static_cast<float*>(p.q), static_cast<float*>(cache.k), static_cast<float*>(cache.v),
                          cache.max_T, d->rope_style, lens)))
    return rc;
  if ((rc = simt_attention(c, static_cast<float*>(p.q), static_cast<float*>(cache.k), static_cast<float*>(cache.v),
                           start, static_cast<float*>(p.o), B, S, H, G, D, cache.max_T, max_pos, lens)))
    return rc;
  if ((rc = simt_linear(c, 1, static_cast<float*>(p.o), static_cast<const float*>(w->wo), nullptr, nullptr, xf, h, M,
                        dm, H * D)))
    return rc;
  if ((rc = rmsnorm(c, h, w->ffn_norm, xn, M, dm, d->rms_eps, d->dtype))) return rc;
  if ((rc = simt_linear(c, 2, xn, static_cast<const float*>(w->w_gate), static_cast<const float*>(w->w_up), nullptr,
                        nullptr, a, M, I, dm)))
    return rc;
  return simt_linear(c, 1, a, static_cast<const float*>(w->w_down), nullptr, nullptr, h, static_cast<float*>(out), M,
                     dm, I);
}

int check_prefill_args(const llama_layer_dims* d, const llama_layer_weights* w, const void* x, const void* out,
                       const float* cos, const float* sin, int max_pos, const llama_kv_cache& cache, int B, int S) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_weights(w))) return rc;
  if (!x || !out || !cos || !sin || !cache.k || !cache.v) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(cos) || !aligned16(sin) || !aligned16(cache.k) ||
      !aligned16(cache.v))
    return LLAMA_ERR_INVALID_ARG;
  if (x == out) return LLAMA_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || max_pos <= 0 || cache.max_T <= 0) return LLAMA_ERR_INVALID_ARG;
  if (S > max_pos || S > cache.max_T) return LLAMA_ERR_INVALID_ARG;
  return LLAMA_OK;
}

// One decode step of one layer; arguments already checked, workspace laid out by decode_ws.
// bf16 layers in a stack: `xn_given` means the workspace's xn already holds RMSNorm₁(x) (the
// previous layer's last kernel wrote it), and a non-null `next_norm` makes this layer's last
// kernel also write RMSNorm(out) with that gamma into xn (the next layer's input norm, or the
// model's final norm).
int decode_impl(const Ctx& c0, const Ctx& c, const llama_layer_dims* dims, const llama_layer_weights* w,
                const void* x, void* out, const float* cos, const float* sin, int32_t max_pos,
                const int32_t* positions, llama_kv_cache cache, int32_t B, void* workspace,
                const void* next_norm = nullptr, bool xn_given = false) {
  int rc;
  DecodeWs p;
  decode_ws(dims, B, cache.max_T, c.num_sms, workspace, &p);
  const int dm = dims->d_model, H = dims->n_heads, G = dims->n_kv_heads, D = dims->head_dim, I = dims->d_inter;
  const int T = cache.max_T;
  if (dims->dtype == LLAMA_BF16) {
    float* P = static_cast<float*>(p.part);
    const int qkv = (H + 2 * G) * D;
    if (!xn_given && (rc = rmsnorm(c0, x, w->attn_norm, p.xn, B, dm, dims->rms_eps, dims->dtype))) return rc;
    {
      const void* W3[3] = {w->wq, w->wk, w->wv};
      const int R3[3] = {H * D, G * D, G * D};
      const int s = choose_splits(c.num_sms, qkv, dm, B);
      if ((rc = gemm_tokens_partial(c, W3, R3, 3, p.xn, B, dm, s, P))) return rc;
      if ((rc = fix_qkv_rope(c, P, s, B, H, G, D, positions, max_pos, cos, sin, p.q, cache.k, cache.v, T,
                             dims->rope_style)))
        return rc;
    }
    if ((rc = attn_decode(c, dims->dtype, p.q, cache.k, cache.v, positions, p.o, B, H, G, D, T, max_pos, p.attn)))
      return rc;
    {
      const void* W1[1] = {w->wo};
      const int R1[1] = {dm};
      const int s = choose_splits(c.num_sms, dm, H * D, B);
      if ((rc = gemm_tokens_partial(c, W1, R1, 1, p.o, B, H * D, s, P))) return rc;
      // h = x + O Wo^T, then the MLP's RMSNorm of h, in one pass over each token's row
      if ((rc = fix_residual_rmsnorm(c, P, s, B, dm, x, w->ffn_norm, dims->rms_eps, p.h, p.xn))) return rc;
    }
    {
      const void* W2[2] = {w->w_gate, w->w_up};
      const int R2[2] = {I, I};
      const int s = choose_splits(c.num_sms, 2 * I, dm, B);
      if ((rc = gemm_tokens_partial(c, W2, R2, 2, p.xn, B, dm, s, P))) return rc;
      if ((rc = fix_swiglu(c, P, s, B, I, p.a))) return rc;
    }
    {
      const void* W1[1] = {w->w_down};
      const int R1[1] = {dm};
      const int s = choose_splits(c.num_sms, dm, I, B);
      if ((rc = gemm_tokens_partial(c, W1, R1, 1, p.a, B, I, s, P))) return rc;
      if (next_norm != nullptr) return fix_residual_rmsnorm(c, P, s, B, dm, p.h, next_norm, dims->rms_eps, out, p.xn);
      return fix_residual(c, P, s, B, dm, p.h, out);
    }
  }
  float* xn = static_cast<float*>(p.xn);
  float* h = static_cast<float*>(p.h);
  float* a = static_cast<float*>(p.a);
  if ((rc = rmsnorm(c0, x, w->attn_norm, xn, B, dm, dims->rms_eps, dims->dtype))) return rc;
  if ((rc = simt_qkv_rope(c, xn, static_cast<const float*>(w->wq), static_cast<const float*>(w->wk),
                          static_cast<const float*>(w->wv), B, 1, dm, H, G, D, cos, sin, positions, max_pos,
                          static_cast<float*>(p.q), static_cast<float*>(cache.k), static_cast<float*>(cache.v), T,
                          dims->rope_style)))
    return rc;
  if ((rc = simt_attention(c, static_cast<float*>(p.q), static_cast<float*>(cache.k), static_cast<float*>(cache.v),
                           positions, static_cast<float*>(p.o), B, 1, H, G, D, T, max_pos)))
    return rc;
  if ((rc = simt_linear(c, 1, static_cast<float*>(p.o), static_cast<const float*>(w->wo), nullptr, nullptr,
                        static_cast<const float*>(x), h, B, dm, H * D)))
    return rc;
  if ((rc = rmsnorm(c, h, w->ffn_norm, xn, B, dm, dims->rms_eps, dims->dtype))) return rc;
  if ((rc = simt_linear(c, 2, xn, static_cast<const float*>(w->w_gate), static_cast<const float*>(w->w_up), nullptr,
                        nullptr, a, B, I, dm)))
    return rc;
  return simt_linear(c, 1, a, static_cast<const float*>(w->w_down), nullptr, nullptr, h, static_cast<float*>(out), B,
                     dm, I);
}

// Workspace of llama_stack_decode: ping-pong activations, one layer's decode workspace and
// the LM head's split-K partials.
struct StackDecodeWs {
  void* xa;
  void* xb;
  void* layer;
  float* part;
};

int lm_head_splits(const llama_stack* st, int B, int num_sms) {
  if (st->dims.dtype != LLAMA_BF16 || st->vocab % 128 != 0) return 0;   // 0: not the weight-streaming form
  return choose_splits(num_sms, st->vocab, st->dims.d_model, B);
}

size_t stack_decode_ws(const llama_stack* st, int B, int num_sms, void* base, StackDecodeWs* out) {
  const llama_layer_dims* d = &st->dims;
  const size_t es = esize(d->dtype);
  Carver cv(base);
  StackDecodeWs w;
  w.xa = cv.take(static_cast<size_t>(B) * d->d_model * es);
  w.xb = cv.take(static_cast<size_t>(B) * d->d_model * es);
  w.layer = cv.take(decode_ws(d, B, 1, num_sms, nullptr, nullptr));
  const int s = lm_head_splits(st, B, num_sms);
  w.part = static_cast<float*>(cv.take(s > 1 ? static_cast<size_t>(s) * B * st->vocab * sizeof(float) : 0));
  if (out) *out = w;
  return cv.off;
}

int check_stack(const llama_stack* st) {
  if (st == nullptr) return LLAMA_ERR_INVALID_ARG;
  int rc = check_dims(&st->dims);
  if (rc) return rc;
  if (st->n_layers < 0 || st->vocab <= 0 || st->final_norm == nullptr || st->embed == nullptr ||
      st->lm_head == nullptr || (st->n_layers > 0 && st->layers == nullptr))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(st->embed) || !aligned16(st->lm_head) || !aligned16(st->final_norm)) return LLAMA_ERR_INVALID_ARG;
  if (st->dims.dtype == LLAMA_BF16 && st->vocab % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  if ((st->dims.d_model * esize(st->dims.dtype)) % 16 != 0) return LLAMA_ERR_UNSUPPORTED;
  return LLAMA_OK;
}

// The contexts of a composite call: its first kernel waits for everything queued before
// the call (no programmatic serialisation), the rest overlap their predecessors; the
// weights are the caller's parameters, so GEMMs may prefetch them.
void call_contexts(const Ctx& base, Ctx* first, Ctx* rest) {
  *rest = base;
  rest->static_weights = true;
  *first = *rest;
  first->pdl = false;
}

// One decode step of the stack; arguments already checked.
int stack_decode_impl(const Ctx& c, const llama_stack* st, const int32_t* tokens, const int32_t* positions,
                      float* logits, const float* cos, const float* sin, int32_t max_pos,
                      const llama_kv_cache* caches, int32_t B, void* workspace) {
  const llama_layer_dims* d = &st->dims;
  const size_t es = esize(d->dtype);
  StackDecodeWs p;
  stack_decode_ws(st, B, c.num_sms, workspace, &p);
  int rc;
  Ctx c0, cr;
  call_contexts(c, &c0, &cr);
  if ((rc = embed_gather(c0, tokens, st->embed, p.xa, B, static_cast<int>(d->d_model * es), st->vocab))) return rc;
  void* xa = p.xa;
  void* xb = p.xb;
  // bf16: each layer's last kernel also normalises its output for what follows (the next
  // layer's attn_norm, the final norm after the last layer) into the layer workspace's xn
  const bool fuse = d->dtype == LLAMA_BF16 && st->n_layers > 0;
  DecodeWs lw;
  decode_ws(d, B, 1, c.num_sms, p.layer, &lw);
  for (int l = 0; l < st->n_layers; ++l) {
    const void* nn = !fuse ? nullptr : l + 1 < st->n_layers ? st->layers[l + 1].attn_norm : st->final_norm;
    if ((rc = decode_impl(cr, cr, d, &st->layers[l], xa, xb, cos, sin, max_pos, positions, caches[l], B, p.layer,
                          nn, fuse && l > 0)))
      return rc;
    std::swap(xa, xb);
  }
  // final RMSNorm (already in the layer workspace when fused), then the untied LM head in fp32
  if (fuse) {
    xb = lw.xn;
  } else if ((rc = rmsnorm(cr, xa, st->final_norm, xb, B, d->d_model, d->rms_eps, d->dtype))) {
    return rc;
  }
  if (d->dtype != LLAMA_BF16)
    return simt_linear(cr, 0, static_cast<const float*>(xb), static_cast<const float*>(st->lm_head), nullptr, nullptr,
                       nullptr, logits, B, st->vocab, d->d_model);
  const int s = lm_head_splits(st, B, c.num_sms);
  if (s == 0) return gemm_plain(cr, xb, st->lm_head, logits, B, st->vocab, d->d_model, true);
  const void* W1[1] = {st->lm_head};
  const int R1[1] = {st->vocab};
  if ((rc = gemm_tokens_partial(cr, W1, R1, 1, xb, B, d->d_model, s, s == 1 ? logits : p.part))) return rc;
  return s == 1 ? LLAMA_OK : fix_sum_f32(cr, p.part, s, B, st->vocab, logits);
}

}  // namespace

extern "C" {

int llama_layer_prefill_workspace_bytes(const llama_layer_dims* dims, int32_t B, int32_t S, size_t* bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (bytes == nullptr || B <= 0 || S <= 0) return LLAMA_ERR_INVALID_ARG;
  *bytes = prefill_ws(dims, B, S, nullptr, nullptr);
  return LLAMA_OK;
}

int llama_layer_prefill(const llama_layer_dims* dims, const llama_layer_weights* w, const void* x, void* out,
                        const float* cos, const float* sin, int32_t max_pos, llama_kv_cache cache, int32_t B,
                        int32_t S, void* workspace, size_t ws_bytes, void* cuda_stream) {
  int rc = check_prefill_args(dims, w, x, out, cos, sin, max_pos, cache, B, S);
  if (rc) return rc;
  if (!workspace || !aligned16(workspace) || ws_bytes < prefill_ws(dims, B, S, nullptr, nullptr))
    return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  Ctx c0, cr;
  call_contexts(c, &c0, &cr);
  return prefill_impl(c0, cr, dims, w, x, out, cos, sin, max_pos, cache, B, S, workspace);
}

int llama_layer_prefill_chunk(const llama_layer_dims* dims, const llama_layer_weights* w, const void* x, void* out,
                              const float* cos, const float* sin, int32_t max_pos, const int32_t* start,
                              const int32_t* lengths, llama_kv_cache cache, int32_t B, int32_t S, void* workspace,
                              size_t ws_bytes, void* cuda_stream) {
  int rc = check_prefill_args(dims, w, x, out, cos, sin, max_pos, cache, B, S);
  if (rc) return rc;
  if (start == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < prefill_ws(dims, B, S, nullptr, nullptr))
    return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  Ctx c0, cr;
  call_contexts(c, &c0, &cr);
  return prefill_impl(c0, cr, dims, w, x, out, cos, sin, max_pos, cache, B, S, workspace, start, lengths);
}

int llama_layer_decode_workspace_bytes(const llama_layer_dims* dims, int32_t B, int32_t max_T, size_t* bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (bytes == nullptr || B <= 0 || max_T <= 0) return LLAMA_ERR_INVALID_ARG;
  int sms = 0;
  if (dims->dtype == LLAMA_BF16 && (rc = num_sms_current(&sms))) return rc;
  *bytes = decode_ws(dims, B, max_T, sms, nullptr, nullptr);
  return LLAMA_OK;
}

int llama_layer_decode(const llama_layer_dims* dims, const llama_layer_weights* w, const void* x, void* out,
                       const float* cos, const float* sin, int32_t max_pos, const int32_t* positions,
                       llama_kv_cache cache, int32_t B, void* workspace, size_t ws_bytes, void* cuda_stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if ((rc = check_weights(w))) return rc;
  if (!x || !out || !cos || !sin || !positions || !cache.k || !cache.v || !workspace) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned16(cos) || !aligned16(sin) || !aligned16(cache.k) ||
      !aligned16(cache.v) || !aligned16(workspace) || x == out)
    return LLAMA_ERR_INVALID_ARG;
  if (B <= 0 || max_pos <= 0 || cache.max_T <= 0) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  if (ws_bytes < decode_ws(dims, B, cache.max_T, c.num_sms, nullptr, nullptr)) return LLAMA_ERR_INVALID_ARG;
  Ctx c0, cr;
  call_contexts(c, &c0, &cr);
  return decode_impl(c0, cr, dims, w, x, out, cos, sin, max_pos, positions, cache, B, workspace);
}

int llama_stack_workspace_bytes(const llama_stack* st, int32_t B, int32_t S, size_t* bytes) {
  if (st == nullptr || bytes == nullptr || B <= 0 || S <= 0) return LLAMA_ERR_INVALID_ARG;
  int rc = check_dims(&st->dims);
  if (rc) return rc;
  const size_t es = esize(st->dims.dtype);
  const size_t M = static_cast<size_t>(B) * S;
  size_t total = 0;
  total += 2 * align_up(M * st->dims.d_model * es);                                           // ping-pong activations
  total += 2 * align_up(M * st->dims.n_kv_heads * st->dims.head_dim * es);                    // K/V if no caches
  total += align_up(prefill_ws(&st->dims, B, S, nullptr, nullptr));
  total += align_up((2 * static_cast<size_t>(st->n_layers) + 1) * sizeof(int));   // the GEMM prologues' counts
  *bytes = total;
  return LLAMA_OK;
}

int llama_stack_forward(const llama_stack* st, const int32_t* tokens, float* logits, const float* cos,
                        const float* sin, int32_t max_pos, const llama_kv_cache* caches, int32_t B, int32_t S,
                        void* workspace, size_t ws_bytes, void* cuda_stream) {
  if (st == nullptr || tokens == nullptr || logits == nullptr || workspace == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (st->n_layers < 0 || st->vocab <= 0 || st->final_norm == nullptr || st->embed == nullptr ||
      st->lm_head == nullptr || (st->n_layers > 0 && st->layers == nullptr))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(logits) || !aligned16(workspace) || !aligned16(st->embed) ||
      !aligned16(st->lm_head) || !aligned16(st->final_norm))
    return LLAMA_ERR_INVALID_ARG;
  size_t need = 0;
  int rc = llama_stack_workspace_bytes(st, B, S, &need);
  if (rc) return rc;
  if (ws_bytes < need) return LLAMA_ERR_INVALID_ARG;
  const llama_layer_dims* d = &st->dims;
  if (d->dtype == LLAMA_BF16 && st->vocab % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  if ((d->d_model * esize(d->dtype)) % 16 != 0) return LLAMA_ERR_UNSUPPORTED;
  const size_t es = esize(d->dtype);
  const size_t M = static_cast<size_t>(B) * S;
  Carver cv(workspace);
  void* xa = cv.take(M * d->d_model * es);
  void* xb = cv.take(M * d->d_model * es);
  void* ks = cv.take(M * d->n_kv_heads * d->head_dim * es);
  void* vs = cv.take(M * d->n_kv_heads * d->head_dim * es);
  void* lws = cv.take(prefill_ws(d, B, S, nullptr, nullptr));
  int* sync = static_cast<int*>(cv.take((2 * static_cast<size_t>(st->n_layers) + 1) * sizeof(int)));
  for (int l = 0; l < st->n_layers; ++l) {
    llama_kv_cache kc = caches ? caches[l] : llama_kv_cache{ks, vs, S};
    if ((rc = check_prefill_args(d, &st->layers[l], xa, xb, cos, sin, max_pos, kc, B, S))) return rc;
  }
  if (st->n_layers == 0 && (S > max_pos || !cos || !sin)) return LLAMA_ERR_INVALID_ARG;
  Ctx c_base, c0, c;
  if ((rc = make_ctx(cuda_stream, &c_base))) return rc;
  call_contexts(c_base, &c0, &c);
  if ((rc = embed_gather(c0, tokens, st->embed, xa, static_cast<int>(M), static_cast<int>(d->d_model * es),
                         st->vocab)))
    return rc;
  // bf16: every RMSNorm runs in the prologue of the GEMM after it, each with its own count
  const bool tc = d->dtype == LLAMA_BF16;
  PrefillWs pw;
  prefill_ws(d, B, S, lws, &pw);
  if (tc && cudaMemsetAsync(sync, 0, (2 * static_cast<size_t>(st->n_layers) + 1) * sizeof(int), c.stream) !=
                cudaSuccess)
    return LLAMA_ERR_CUDA;
  for (int l = 0; l < st->n_layers; ++l) {
    llama_kv_cache kc = caches ? caches[l] : llama_kv_cache{ks, vs, S};
    if ((rc = prefill_impl(c, c, d, &st->layers[l], xa, xb, cos, sin, max_pos, kc, B, S, lws, nullptr, nullptr,
                           tc ? sync + 2 * l : nullptr)))
      return rc;
    void* t = xa;
    xa = xb;
    xb = t;
  }
  // final RMSNorm (required by the pre-norm layout), then the untied LM head in fp32; bf16
  // stacks normalise in the LM head GEMM's prologue
  if (tc) {
    const NormPro fn{st->final_norm, d->rms_eps, pw.xn, sync + 2 * st->n_layers};
    return gemm_plain(c, xa, st->lm_head, logits, static_cast<int>(M), st->vocab, d->d_model, true, &fn);
  }
  if ((rc = rmsnorm(c, xa, st->final_norm, xb, static_cast<int>(M), d->d_model, d->rms_eps, d->dtype))) return rc;
  return simt_linear(c, 0, static_cast<const float*>(xb), static_cast<const float*>(st->lm_head), nullptr, nullptr,
                     nullptr, logits, static_cast<int>(M), st->vocab, d->d_model);
}

int llama_stack_decode_workspace_bytes(const llama_stack* st, int32_t B, size_t* bytes) {
  int rc = check_stack(st);
  if (rc) return rc;
  if (bytes == nullptr || B <= 0) return LLAMA_ERR_INVALID_ARG;
  int sms = 0;
  if (st->dims.dtype == LLAMA_BF16 && (rc = num_sms_current(&sms))) return rc;
  *bytes = stack_decode_ws(st, B, sms, nullptr, nullptr);
  return LLAMA_OK;
}

int llama_stack_decode(const llama_stack* st, const int32_t* tokens, const int32_t* positions, float* logits,
                       const float* cos, const float* sin, int32_t max_pos, const llama_kv_cache* caches, int32_t B,
                       void* workspace, size_t ws_bytes, void* cuda_stream) {
  int rc = check_stack(st);
  if (rc) return rc;
  if (!tokens || !positions || !logits || !cos || !sin || !workspace || B <= 0 || max_pos <= 0) return LLAMA_ERR_INVALID_ARG;
  if (st->n_layers > 0 && caches == nullptr) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(logits) || !aligned16(workspace) || !aligned16(cos) || !aligned16(sin))
    return LLAMA_ERR_INVALID_ARG;
  for (int l = 0; l < st->n_layers; ++l) {
    if ((rc = check_weights(&st->layers[l]))) return rc;
    const llama_kv_cache& kc = caches[l];
    if (!kc.k || !kc.v || kc.max_T <= 0 || !aligned16(kc.k) || !aligned16(kc.v)) return LLAMA_ERR_INVALID_ARG;
  }
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  if (ws_bytes < stack_decode_ws(st, B, c.num_sms, nullptr, nullptr)) return LLAMA_ERR_INVALID_ARG;
  return stack_decode_impl(c, st, tokens, positions, logits, cos, sin, max_pos, caches, B, workspace);
}

int llama_rmsnorm(const void* x, const void* gamma, void* y, int32_t rows, int32_t d, float eps, int32_t dtype,
                  void* cuda_stream) {
  if (!x || !gamma || !y || rows < 0 || d <= 0 || !(eps >= 0.f) || (dtype != LLAMA_F32 && dtype != LLAMA_BF16))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma)) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  return rmsnorm(c, x, gamma, y, rows, d, eps, dtype);
}

int llama_layernorm(const void* x, const void* gamma, const void* beta, void* y, int32_t rows, int32_t d, float eps,
                    int32_t dtype, void* cuda_stream) {
  if (!x || !gamma || !beta || !y || rows < 0 || d <= 0 || !(eps >= 0.f) || (dtype != LLAMA_F32 && dtype != LLAMA_BF16))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta)) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  return layernorm(c, x, gamma, beta, y, rows, d, eps, dtype);
}

int llama_linear_bf16(const void* A, const void* B, void* C, int32_t M, int32_t N, int32_t K, int32_t c_f32,
                      void* cuda_stream) {
  if (!A || !B || !C || M <= 0 || N <= 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  return gemm_plain(c, A, B, C, M, N, K, c_f32 != 0);
}

int llama_linear_residual(const void* A, const void* W, const void* resid, void* out, int32_t M, int32_t N, int32_t K,
                          void* cuda_stream) {
  if (!A || !W || !resid || !out || M <= 0 || N <= 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(resid) || !aligned16(out)) return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 128 != 0) return LLAMA_ERR_UNSUPPORTED;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  return gemm_residual(c, A, W, resid, out, M, N, K);
}

int llama_linear_swiglu(const void* A, const void* W_gate, const void* W_up, void* out, int32_t M, int32_t I, int32_t K,
                        void* cuda_stream) {
  if (!A || !W_gate || !W_up || !out || M <= 0 || I <= 0 || K <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(out)) return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || I % 128 != 0) return LLAMA_ERR_UNSUPPORTED;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  return gemm_swiglu(c, A, W_gate, W_up, out, M, I, K);
}

int llama_qkv_rope(const llama_layer_dims* dims, const void* xn, const void* wq, const void* wk, const void* wv,
                   const float* cos, const float* sin, int32_t max_pos, llama_kv_cache cache, void* q_out, int32_t B,
                   int32_t S, void* cuda_stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (dims->dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (!xn || !wq || !wk || !wv || !cos || !sin || !cache.k || !cache.v || !q_out) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(cache.k) ||
      !aligned16(cache.v) || !aligned16(q_out))
    return LLAMA_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || S > max_pos || S > cache.max_T) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  return gemm_qkv_rope(c, xn, wq, wk, wv, B, S, dims->d_model, dims->n_heads, dims->n_kv_heads, dims->head_dim, cos,
                       sin, q_out, cache.k, cache.v, cache.max_T, dims->rope_style);
}

int llama_layer_prefill_workspace_layout(const llama_layer_dims* dims, int32_t B, int32_t S, size_t* offsets) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (offsets == nullptr || B <= 0 || S <= 0) return LLAMA_ERR_INVALID_ARG;
  // carve a workspace at a stand-in base address (never dereferenced) and subtract it
  uint8_t* const base = reinterpret_cast<uint8_t*>(kAlign);
  PrefillWs w;
  prefill_ws(dims, B, S, base, &w);
  const void* regions[5] = {w.q, w.o, w.h, w.a, w.xn};
  for (int i = 0; i < 5; ++i) offsets[i] = static_cast<size_t>(static_cast<const uint8_t*>(regions[i]) - base);
  return LLAMA_OK;
}

int llama_stack_workspace_layout(const llama_stack* st, int32_t B, int32_t S, size_t* offsets) {
  if (st == nullptr || offsets == nullptr || B <= 0 || S <= 0 || st->n_layers < 0) return LLAMA_ERR_INVALID_ARG;
  int rc = check_dims(&st->dims);
  if (rc) return rc;
  // the carve-up of llama_stack_forward: two activation buffers (the layers ping-pong between
  // them), the workspace's own K/V, the layer workspace
  const size_t es = esize(st->dims.dtype);
  const size_t M = static_cast<size_t>(B) * S;
  Carver cv(reinterpret_cast<void*>(kAlign));
  uint8_t* act[2];
  act[0] = static_cast<uint8_t*>(cv.take(M * st->dims.d_model * es));
  act[1] = static_cast<uint8_t*>(cv.take(M * st->dims.d_model * es));
  cv.take(M * st->dims.n_kv_heads * st->dims.head_dim * es);
  cv.take(M * st->dims.n_kv_heads * st->dims.head_dim * es);
  uint8_t* lws = static_cast<uint8_t*>(cv.take(prefill_ws(&st->dims, B, S, nullptr, nullptr)));
  const int n = st->n_layers;
  uint8_t* const base = reinterpret_cast<uint8_t*>(kAlign);
  offsets[0] = static_cast<size_t>(act[n % 2 == 1 ? 0 : 1] - base);   // the last layer's input
  offsets[1] = static_cast<size_t>(act[n % 2] - base);                // its output
  offsets[2] = static_cast<size_t>(lws - base);
  return LLAMA_OK;
}

int llama_norm_linear_bf16(const void* A, const void* gamma, float eps, const void* B, void* C, int32_t M, int32_t N,
                           int32_t K, int32_t c_f32, void* xn, int32_t* sync, void* cuda_stream) {
  if (!A || !gamma || !B || !C || !xn || !sync || M <= 0 || N <= 0 || K <= 0 || !(eps >= 0.f))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(gamma) || !aligned16(B) || !aligned16(C) || !aligned16(xn) || A == xn)
    return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  if (cudaMemsetAsync(sync, 0, sizeof(int), c.stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  const NormPro n{gamma, eps, xn, sync};
  return gemm_plain(c, A, B, C, M, N, K, c_f32 != 0, &n);
}

int llama_norm_linear_swiglu(const void* A, const void* gamma, float eps, const void* W_gate, const void* W_up,
                             void* out, int32_t M, int32_t I, int32_t K, void* xn, int32_t* sync, void* cuda_stream) {
  if (!A || !gamma || !W_gate || !W_up || !out || !xn || !sync || M <= 0 || I <= 0 || K <= 0 || !(eps >= 0.f))
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(gamma) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(out) ||
      !aligned16(xn) || A == xn)
    return LLAMA_ERR_INVALID_ARG;
  if (K % 8 != 0 || I % 128 != 0) return LLAMA_ERR_UNSUPPORTED;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc) return rc;
  if (cudaMemsetAsync(sync, 0, sizeof(int), c.stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  const NormPro n{gamma, eps, xn, sync};
  return gemm_swiglu(c, A, W_gate, W_up, out, M, I, K, &n);
}

int llama_norm_qkv_rope(const llama_layer_dims* dims, const void* x, const void* attn_norm, const void* wq,
                        const void* wk, const void* wv, const float* cos, const float* sin, int32_t max_pos,
                        llama_kv_cache cache, void* q_out, int32_t B, int32_t S, void* xn, int32_t* sync,
                        void* cuda_stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (dims->dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (!x || !attn_norm || !wq || !wk || !wv || !cos || !sin || !cache.k || !cache.v || !q_out || !xn || !sync)
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(attn_norm) || !aligned16(wq) || !aligned16(wk) || !aligned16(wv) ||
      !aligned16(cos) || !aligned16(sin) || !aligned16(cache.k) || !aligned16(cache.v) || !aligned16(q_out) ||
      !aligned16(xn) || x == xn)
    return LLAMA_ERR_INVALID_ARG;
  if (B <= 0 || S <= 0 || S > max_pos || S > cache.max_T) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  if (cudaMemsetAsync(sync, 0, sizeof(int), c.stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  const NormPro n{attn_norm, dims->rms_eps, xn, sync};
  return gemm_qkv_rope(c, x, wq, wk, wv, B, S, dims->d_model, dims->n_heads, dims->n_kv_heads, dims->head_dim, cos,
                       sin, q_out, cache.k, cache.v, cache.max_T, dims->rope_style, nullptr, nullptr, max_pos, &n);
}

int llama_attention_prefill(const llama_layer_dims* dims, const void* q, llama_kv_cache cache, void* out, int32_t B,
                            int32_t S, void* cuda_stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!q || !out || !cache.k || !cache.v || B <= 0 || S <= 0 || S > cache.max_T) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(cache.k) || !aligned16(cache.v)) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  if (dims->dtype == LLAMA_BF16)
    return attn_prefill_tc(c, q, cache.k, cache.v, out, B, S, dims->n_heads, dims->n_kv_heads, dims->head_dim,
                           cache.max_T);
  return simt_attention(c, static_cast<const float*>(q), static_cast<const float*>(cache.k),
                        static_cast<const float*>(cache.v), nullptr, static_cast<float*>(out), B, S, dims->n_heads,
                        dims->n_kv_heads, dims->head_dim, cache.max_T, cache.max_T);
}

int llama_attention_decode_workspace_bytes(const llama_layer_dims* dims, int32_t B, int32_t max_T, size_t* bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!bytes || B <= 0 || max_T <= 0) return LLAMA_ERR_INVALID_ARG;
  *bytes = attn_decode_ws_bytes(B, dims->n_heads, dims->n_kv_heads, dims->head_dim);
  return LLAMA_OK;
}

int llama_attention_decode(const llama_layer_dims* dims, const void* q, llama_kv_cache cache,
                           const int32_t* positions, void* out, int32_t B, void* workspace, size_t ws_bytes,
                           void* cuda_stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!q || !out || !cache.k || !cache.v || !positions || B <= 0 || cache.max_T <= 0) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(cache.k) || !aligned16(cache.v)) return LLAMA_ERR_INVALID_ARG;
  Ctx c;
  if ((rc = make_ctx(cuda_stream, &c))) return rc;
  if (dims->dtype == LLAMA_BF16) {
    if (!workspace || !aligned16(workspace) ||
        ws_bytes < attn_decode_ws_bytes(B, dims->n_heads, dims->n_kv_heads, dims->head_dim))
      return LLAMA_ERR_INVALID_ARG;
    return attn_decode(c, dims->dtype, q, cache.k, cache.v, positions, out, B, dims->n_heads, dims->n_kv_heads,
                       dims->head_dim, cache.max_T, cache.max_T, workspace);
  }
  return simt_attention(c, static_cast<const float*>(q), static_cast<const float*>(cache.k),
                        static_cast<const float*>(cache.v), positions, static_cast<float*>(out), B, 1, dims->n_heads,
                        dims->n_kv_heads, dims->head_dim, cache.max_T, cache.max_T);
}

}  // extern "C"
