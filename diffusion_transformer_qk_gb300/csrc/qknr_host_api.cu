// The fused QK-RMSNorm + RoPE from host-resident activations
// (qknr_forward_host): token rows go through caller-owned device staging
// buffers in chunks, with the host-to-device copy of one chunk, the kernel
// on the previous one and the device-to-host copy of the one before that on
// three streams.  Each chunk is one qknr_forward on its staging buffer, in
// place, so every row sees the same kernel and table row as one call over
// the whole activation.  No allocation: buffers, streams and events belong
// to the caller.
#include <cuda_runtime.h>

#include <cstring>

#include "../../include/qknr.h"
#include "qknr_host.h"

namespace {

using qknr_host::cuda_fail;
using qknr_host::fail;
using qknr_host::overlaps;
using qknr_host::Span;
using qknr_host::span_of;

// One host tensor's columns of a chunk: `heads` heads at `base` with a row
// stride of `stride` elements.
struct HostSlice {
  const char* base;
  long long stride_bytes;
  long long bytes;                 // heads * D * 2 per row
};

// A 2-D copy of `rows` rows of `width` bytes between pitched buffers.
qknr_status copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, long long rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (rows <= 0 || width == 0) return QKNR_OK;
  const cudaError_t e = cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, static_cast<size_t>(rows), kind, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
  return QKNR_OK;
}

struct Pipe {
  long long T = 0, chunk = 0, cos_rows = 0, cos_row_bytes = 0;
  int D = 0, hq = 0, hk = 0, hv = 0;   // hv: V heads carried through (copied), else 0
  long long width = 0;                 // staging row bytes: (hq + hk + hv) * D * 2
  // host inputs and outputs of Q, K and (when copied) V, and whether each
  // tensor follows the previous one in the same host rows (one copy for both)
  HostSlice in[3], out[3];
  bool in_joined[3], out_joined[3];
  bool per_token_table = true;         // cos_rows >= tokens: chunks take their own table rows
};

qknr_status plan_pipe(const qknr_args* a, const qknr_host_plan* p, Pipe* pp) {
  if (!a || !p) return fail(QKNR_ERR_NULL, "args or plan is NULL");
  if (a->abi_version != QKNR_ABI_VERSION || p->abi_version != QKNR_ABI_VERSION)
    return fail(QKNR_ERR_ABI, "abi_version mismatch (library expects %d)", QKNR_ABI_VERSION);
  if (p->n_buffers < 1 || p->n_buffers > QKNR_HOST_MAX_BUFFERS)
    return fail(QKNR_ERR_SHAPE, "n_buffers must be 1..%d", QKNR_HOST_MAX_BUFFERS);
  if (p->chunk_rows <= 0) return fail(QKNR_ERR_SHAPE, "chunk_rows must be > 0");
  if (a->dtype != QKNR_BF16 && a->dtype != QKNR_FP16)
    return fail(QKNR_ERR_UNSUPPORTED, "activation dtype must be BF16 or FP16");
  if (a->head_dim != 64 && a->head_dim != 128)
    return fail(QKNR_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", a->head_dim);
  if (a->tokens < 0 || a->n_heads_q < 0 || a->n_heads_k < 0 || a->n_heads_v < 0 || a->cos_rows < 0)
    return fail(QKNR_ERR_SHAPE, "negative size");
  Pipe& P = *pp;
  P.T = a->tokens;
  P.chunk = p->chunk_rows;
  P.D = a->head_dim;
  P.hq = a->n_heads_q;
  P.hk = a->n_heads_k;
  const long long es = 2, D = P.D;
  const long long qs = a->q_stride ? a->q_stride : P.hq * D;
  const long long ks = a->k_stride ? a->k_stride : P.hk * D;
  const long long vs = a->v_stride ? a->v_stride : a->n_heads_v * D;
  const long long qos = a->q_out_stride ? a->q_out_stride : qs;
  const long long kos = a->k_out_stride ? a->k_out_stride : ks;
  const long long vos = a->v_out_stride ? a->v_out_stride : vs;
  const bool copy_v = a->n_heads_v > 0 && a->v_out && !(a->v_out == a->v && vos == vs);
  P.hv = copy_v ? a->n_heads_v : 0;
  P.width = (P.hq + P.hk + P.hv) * D * es;
  if (P.hq > 0 && (!a->q || qs < P.hq * D || qos < P.hq * D))
    return fail(P.hq && !a->q ? QKNR_ERR_NULL : QKNR_ERR_SHAPE, "q missing or q strides too small");
  if (P.hk > 0 && (!a->k || ks < P.hk * D || kos < P.hk * D))
    return fail(P.hk && !a->k ? QKNR_ERR_NULL : QKNR_ERR_SHAPE, "k missing or k strides too small");
  if (P.hv > 0 && (!a->v || vs < P.hv * D || vos < P.hv * D))
    return fail(!a->v ? QKNR_ERR_NULL : QKNR_ERR_SHAPE, "v missing or v strides too small");
  const char* q_out = static_cast<const char*>(a->q_out ? a->q_out : a->q);
  const char* k_out = static_cast<const char*>(a->k_out ? a->k_out : a->k);
  P.in[0] = {static_cast<const char*>(a->q), qs * es, P.hq * D * es};
  P.in[1] = {static_cast<const char*>(a->k), ks * es, P.hk * D * es};
  P.in[2] = {static_cast<const char*>(a->v), vs * es, P.hv * D * es};
  P.out[0] = {q_out, qos * es, P.hq * D * es};
  P.out[1] = {k_out, kos * es, P.hk * D * es};
  P.out[2] = {static_cast<const char*>(a->v_out), vos * es, P.hv * D * es};
  for (int side = 0; side < 2; ++side) {
    HostSlice* h = side ? P.out : P.in;
    bool* joined = side ? P.out_joined : P.in_joined;
    joined[0] = false;
    for (int i = 1; i < 3; ++i) {
      // tensor i continues the previous non-empty one in the same rows
      int j = i - 1;
      while (j >= 0 && h[j].bytes == 0) --j;
      joined[i] = h[i].bytes > 0 && j >= 0 && h[i].base == h[j].base + h[j].bytes &&
                  h[i].stride_bytes == h[j].stride_bytes;
    }
  }
  // an output that is not exactly its own input must not overlap any input
  if (P.T > 0) {
    Span ins[3], outs[3];
    for (int i = 0; i < 3; ++i) {
      ins[i] = span_of(P.in[i].base, P.in[i].bytes ? P.T : 0, P.in[i].stride_bytes, P.in[i].bytes);
      outs[i] = span_of(P.out[i].base, P.out[i].bytes ? P.T : 0, P.out[i].stride_bytes, P.out[i].bytes);
    }
    for (int i = 0; i < 3; ++i) {
      if (P.out[i].bytes == 0) continue;
      if (P.out[i].base == P.in[i].base && P.out[i].stride_bytes == P.in[i].stride_bytes) continue;
      for (int j = 0; j < 3; ++j)
        if (overlaps(outs[i], ins[j]))
          return fail(QKNR_ERR_OVERLAP, "a host output overlaps a host input without being in place");
    }
  }
  // table rows per chunk
  const int ces = a->cos_dtype == QKNR_FP32 ? 4 : 2;
  const int table_heads = a->cos_layout == QKNR_COS_PER_HEAD_EXPANDED ? (P.hq > P.hk ? P.hq : P.hk) : 1;
  P.cos_row_bytes = static_cast<long long>(table_heads) * D * ces;
  P.cos_rows = a->cos_rows ? a->cos_rows : P.T;
  P.per_token_table = P.cos_rows >= P.T;
  if (!P.per_token_table && P.chunk % P.cos_rows)
    return fail(QKNR_ERR_SHAPE, "chunk_rows %lld is not a multiple of the batch-broadcast table's %lld rows",
                P.chunk, P.cos_rows);
  // staging buffers and events
  for (int b = 0; b < p->n_buffers; ++b) {
    if (!p->dev_buffers[b]) return fail(QKNR_ERR_NULL, "dev_buffers[%d] is NULL", b);
    if (!qknr_host::aligned16(p->dev_buffers[b])) return fail(QKNR_ERR_ALIGN, "dev_buffers[%d] not 16-byte aligned", b);
  }
  for (int i = 0; i < QKNR_HOST_EVENTS(p->n_buffers); ++i)
    if (!p->events[i]) return fail(QKNR_ERR_NULL, "events[%d] is NULL", i);
  return QKNR_OK;
}

// The qknr_forward arguments of chunk [r0, r0 + rows) on staging buffer `buf`.
qknr_args chunk_args(const qknr_args* a, const Pipe& P, void* buf, long long r0, long long rows) {
  qknr_args c = *a;
  char* b = static_cast<char*>(buf);
  const long long es = 2, D = P.D;
  const long long stride = P.width / es;
  c.q = P.hq ? b : nullptr;
  c.k = P.hk ? b + P.hq * D * es : nullptr;
  c.v = nullptr;
  c.q_out = c.k_out = c.v_out = nullptr;             // in place in the staging buffer
  c.q_stride = c.k_stride = c.q_out_stride = c.k_out_stride = stride;
  c.v_stride = c.v_out_stride = 0;
  c.n_heads_v = 0;                                   // V only rides through the staging buffer
  c.tokens = rows;
  if (P.per_token_table) {
    c.cos = static_cast<const char*>(a->cos) + r0 * P.cos_row_bytes;
    c.sin = static_cast<const char*>(a->sin) + r0 * P.cos_row_bytes;
    c.cos_rows = rows;
  }
  return c;
}

// Copy the present tensors of chunk rows [r0, r0 + rows) between the host
// slices and the staging buffer (columns Q | K | V), joined where adjacent.
qknr_status copy_chunk(const Pipe& P, const HostSlice* h, const bool* joined, char* buf, long long r0, long long rows,
                       bool to_device, cudaStream_t s) {
  long long col = 0;                                 // byte column in the staging row
  for (int i = 0; i < 3;) {
    if (h[i].bytes == 0) {
      ++i;
      continue;
    }
    long long bytes = h[i].bytes;
    int j = i + 1;
    while (j < 3 && (h[j].bytes == 0 || joined[j])) bytes += h[j++].bytes;
    char* host = const_cast<char*>(h[i].base) + r0 * h[i].stride_bytes;
    const qknr_status st =
        to_device ? copy_rows(buf + col, P.width, host, h[i].stride_bytes, bytes, rows, cudaMemcpyHostToDevice, s)
                  : copy_rows(host, h[i].stride_bytes, buf + col, P.width, bytes, rows, cudaMemcpyDeviceToHost, s);
    if (st != QKNR_OK) return st;
    col += bytes;
    i = j;
  }
  return QKNR_OK;
}

qknr_status record(cudaEvent_t e, cudaStream_t s) {
  const cudaError_t r = cudaEventRecord(e, s);
  return r == cudaSuccess ? QKNR_OK : cuda_fail(r, "cudaEventRecord");
}

qknr_status wait(cudaStream_t s, cudaEvent_t e) {
  const cudaError_t r = cudaStreamWaitEvent(s, e, 0);
  return r == cudaSuccess ? QKNR_OK : cuda_fail(r, "cudaStreamWaitEvent");
}

}  // namespace

extern "C" {

void qknr_host_plan_init(qknr_host_plan* p) {
  if (!p) return;
  memset(p, 0, sizeof(*p));
  p->abi_version = QKNR_ABI_VERSION;
  p->n_buffers = 3;
  p->chunk_rows = 2048;
}

size_t qknr_sizeof_host_plan(void) { return sizeof(qknr_host_plan); }

qknr_status qknr_host_buffer_bytes(const qknr_args* args, const qknr_host_plan* plan, size_t* bytes) {
  if (!bytes) return fail(QKNR_ERR_NULL, "bytes is NULL");
  *bytes = 0;
  if (!args || !plan) return fail(QKNR_ERR_NULL, "args or plan is NULL");
  if (plan->chunk_rows <= 0) return fail(QKNR_ERR_SHAPE, "chunk_rows must be > 0");
  const long long D = args->head_dim;
  const bool copy_v = args->n_heads_v > 0 && args->v_out &&
                      !(args->v_out == args->v && (args->v_out_stride == 0 || args->v_out_stride == args->v_stride));
  const long long heads = static_cast<long long>(args->n_heads_q) + args->n_heads_k + (copy_v ? args->n_heads_v : 0);
  if (D <= 0 || heads < 0) return fail(QKNR_ERR_SHAPE, "head_dim or head counts out of range");
  *bytes = static_cast<size_t>(plan->chunk_rows * heads * D * 2);
  return QKNR_OK;
}

qknr_status qknr_forward_host(const qknr_args* args, const qknr_host_plan* plan, qknr_stream_t stream) {
  Pipe P;
  qknr_status st = plan_pipe(args, plan, &P);
  if (st != QKNR_OK) return st;
  if (P.T == 0 || P.hq + P.hk + P.hv == 0) return QKNR_OK;
  // validate the launch of a full chunk before anything is enqueued
  {
    qknr_launch_info info;
    const long long rows = P.T < P.chunk ? P.T : P.chunk;
    qknr_args c = chunk_args(args, P, plan->dev_buffers[0], 0, rows);
    st = qknr_query(&c, &info);
    if (st != QKNR_OK) return st;
  }
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaStream_t h2d = reinterpret_cast<cudaStream_t>(plan->h2d_stream);
  const cudaStream_t d2h = reinterpret_cast<cudaStream_t>(plan->d2h_stream);
  const int nb = plan->n_buffers;
  cudaEvent_t ev[QKNR_HOST_EVENTS(QKNR_HOST_MAX_BUFFERS)];
  for (int i = 0; i < QKNR_HOST_EVENTS(nb); ++i) ev[i] = reinterpret_cast<cudaEvent_t>(plan->events[i]);
  cudaEvent_t* loaded = ev;                          // [nb]: chunk copied in
  cudaEvent_t* computed = ev + nb;                   // [nb]: kernel done
  cudaEvent_t* freed = ev + 2 * nb;                  // [nb]: chunk copied out, buffer free
  const cudaEvent_t start = ev[3 * nb], done = ev[3 * nb + 1];

  // the copies come after the work already on the call's stream (device
  // tables it wrote, the previous call's use of the staging buffers)
  if ((st = record(start, s)) != QKNR_OK || (st = wait(h2d, start)) != QKNR_OK || (st = wait(d2h, start)) != QKNR_OK)
    return st;
  const long long D = P.D;
  // the gains, and a batch-broadcast table, go in first; a per-token table
  // goes in with each chunk, its rows ahead of the chunk's activation
  const void* host_tab[4] = {plan->host_gamma_q, plan->host_gamma_k, plan->host_cos, plan->host_sin};
  const void* dev_tab[4] = {args->gamma_q, args->gamma_k, args->cos, args->sin};
  const long long tab_bytes[4] = {D * 4, D * 4, P.cos_rows * P.cos_row_bytes, P.cos_rows * P.cos_row_bytes};
  for (int i = 0; i < 4; ++i)
    if (host_tab[i] && !dev_tab[i]) return fail(QKNR_ERR_NULL, "a host table is given but its device pointer is NULL");
  auto copy_table = [&](int i, long long off, long long bytes) -> qknr_status {
    const cudaError_t e = cudaMemcpyAsync(const_cast<char*>(static_cast<const char*>(dev_tab[i])) + off,
                                          static_cast<const char*>(host_tab[i]) + off, static_cast<size_t>(bytes),
                                          cudaMemcpyHostToDevice, h2d);
    return e == cudaSuccess ? QKNR_OK : cuda_fail(e, "cudaMemcpyAsync(table)");
  };
  for (int i = 0; i < 4; ++i)
    if (host_tab[i] && (i < 2 || !P.per_token_table) && (st = copy_table(i, 0, tab_bytes[i])) != QKNR_OK) return st;
  // Chunk sizes: with a per-token table the first chunks ramp up (1/8, 1/4,
  // 1/2 of chunk_rows) and the last ones ramp down the same way, so that
  // the copy in of the first chunk and the copy out of the last, which
  // nothing overlaps, are short; in between, chunk_rows each.  (A
  // batch-broadcast table needs every chunk to start on a multiple of its
  // rows: chunk_rows each.)
  const long long C = P.chunk, c8 = C / 8;
  const bool ramp = P.per_token_table && c8 >= 8 && P.T >= 4 * C;
  const long long head_end = 7 * c8, tail_start = P.T - 8 * c8;
  auto chunk_rows_at = [&](long long r0) -> long long {
    if (ramp && r0 < head_end) return r0 == 0 ? c8 : (r0 == c8 ? 2 * c8 : 4 * c8);
    if (ramp && r0 >= tail_start) {
      const long long k = r0 - tail_start;
      return k == 0 ? 4 * c8 : (k == 4 * c8 ? 2 * c8 : c8);
    }
    const long long end = ramp ? tail_start : P.T;
    return end - r0 < C ? end - r0 : C;
  };
  long long i = 0;
  for (long long r0 = 0; r0 < P.T; ++i) {
    const long long rows = chunk_rows_at(r0);
    const int b = static_cast<int>(i % nb);
    char* buf = static_cast<char*>(plan->dev_buffers[b]);
    // in: after this buffer's previous chunk has been copied out
    if (i >= nb && (st = wait(h2d, freed[b])) != QKNR_OK) return st;
    if (P.per_token_table)
      for (int t = 2; t < 4; ++t)
        if (host_tab[t] && (st = copy_table(t, r0 * P.cos_row_bytes, rows * P.cos_row_bytes)) != QKNR_OK) return st;
    if ((st = copy_chunk(P, P.in, P.in_joined, buf, r0, rows, true, h2d)) != QKNR_OK) return st;
    if ((st = record(loaded[b], h2d)) != QKNR_OK || (st = wait(s, loaded[b])) != QKNR_OK) return st;
    // the kernel, in place in the staging buffer
    qknr_args c = chunk_args(args, P, buf, r0, rows);
    if ((st = qknr_forward(&c, stream)) != QKNR_OK) return st;
    if ((st = record(computed[b], s)) != QKNR_OK || (st = wait(d2h, computed[b])) != QKNR_OK) return st;
    // out
    if ((st = copy_chunk(P, P.out, P.out_joined, buf, r0, rows, false, d2h)) != QKNR_OK) return st;
    if ((st = record(freed[b], d2h)) != QKNR_OK) return st;
    r0 += rows;
  }
  // the call's stream sees the results once every copy out is done
  if ((st = record(done, d2h)) != QKNR_OK) return st;
  return wait(s, done);
}

}  // extern "C"
