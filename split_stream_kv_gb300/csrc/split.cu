// split.cu -- the split-stream transfer of "Lynx: Progressive Speculative KV
// Cache Transfer for Disaggregated LLM Inference" (technical review,
// Mechanism 2 and Figure 4; Implementation Notes): a schedule of copies and
// kernels over page groups, and the two executors that enqueue it on CUDA
// streams, plus the serialized-request header.
//
// One GPU plays the role of either side of the link: the sender encodes
// page groups and copies their streams to host memory, the receiver copies
// them from host memory to the device and decodes them.  Every Anchor and
// meta copy is issued before the first Residual copy on one copy queue,
// which is the pages' rule that Anchor buffers are drained before Residual
// buffers at the page level, taken strictly.  (CUDA stream priorities order
// kernels, not copy engines, so the order of the copy queue is what gives
// the Anchor stream its priority.)  Kernels go through the public entry
// points on page ranges: the streams and the BF16 tensor are stored in
// (b, page, head) order, so a range of whole pages is one contiguous slice
// of each, and B = 1, L = pages * page addresses it.
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <vector>

#include "internal.h"
#include "lynx.h"

namespace lynx {
namespace {

struct Dims {
  int64_t B, L;
  int H, D, page, C;
  int64_t ppg;                 // pages per group
  int64_t pages() const { return B * (L / page); }
  int64_t groups() const { return (pages() + ppg - 1) / ppg; }
  int64_t anchor_pp() const { return (int64_t)H * page * (D / 2); }   // bytes per page
  int64_t meta_pp() const { return (int64_t)H * (2 + 2 * (page / C)) * D * 4; }
  int64_t bf16_pp() const { return (int64_t)H * page * D * 2; }
};

lynx_split_op make_op(int kind, int queue, int64_t g, const Dims& d) {
  lynx_split_op op;
  memset(&op, 0, sizeof op);
  op.kind = kind;
  op.queue = queue;
  op.group = g;
  op.page0 = g * d.ppg;
  op.n_pages = d.pages() - op.page0 < d.ppg ? d.pages() - op.page0 : d.ppg;
  op.wait_kind[0] = op.wait_kind[1] = LYNX_OP_NONE;
  op.wait_group[0] = op.wait_group[1] = 0;
  if (kind == LYNX_OP_COPY_ANCHOR || kind == LYNX_OP_COPY_RESIDUAL) {
    op.offset = op.page0 * d.anchor_pp();
    op.bytes = op.n_pages * d.anchor_pp();
  } else if (kind == LYNX_OP_COPY_META) {
    op.offset = op.page0 * d.meta_pp();
    op.bytes = op.n_pages * d.meta_pp();
  }
  return op;
}

void add_wait(lynx_split_op& op, int kind, int64_t group) {
  const int i = op.wait_kind[0] == LYNX_OP_NONE ? 0 : 1;
  op.wait_kind[i] = kind;
  op.wait_group[i] = group;
}

// The schedule, in issue order (every wait names an earlier operation).
std::vector<lynx_split_op> build_plan(const Dims& d, bool send, bool with_decode) {
  std::vector<lynx_split_op> ops;
  const int64_t G = d.groups();
  if (send) {
    for (int64_t g = 0; g < G; ++g) {
      ops.push_back(make_op(LYNX_OP_ENCODE, LYNX_Q_HI, g, d));
      lynx_split_op a = make_op(LYNX_OP_COPY_ANCHOR, LYNX_Q_COPY, g, d);
      add_wait(a, LYNX_OP_ENCODE, g);
      ops.push_back(a);
      ops.push_back(make_op(LYNX_OP_COPY_META, LYNX_Q_COPY, g, d));
    }
    for (int64_t g = 0; g < G; ++g) ops.push_back(make_op(LYNX_OP_COPY_RESIDUAL, LYNX_Q_COPY, g, d));
    return ops;
  }
  for (int64_t g = 0; g < G; ++g) {
    ops.push_back(make_op(LYNX_OP_COPY_ANCHOR, LYNX_Q_COPY, g, d));
    ops.push_back(make_op(LYNX_OP_COPY_META, LYNX_Q_COPY, g, d));
    if (with_decode) {
      lynx_split_op k = make_op(LYNX_OP_DECODE_ANCHOR, LYNX_Q_HI, g, d);
      add_wait(k, LYNX_OP_COPY_META, g);  // the copy queue is in order: anchor g landed too
      ops.push_back(k);
    }
  }
  for (int64_t g = 0; g < G; ++g) {
    ops.push_back(make_op(LYNX_OP_COPY_RESIDUAL, LYNX_Q_COPY, g, d));
    if (with_decode) {
      lynx_split_op u = make_op(LYNX_OP_UPGRADE, LYNX_Q_LO, g, d);
      add_wait(u, LYNX_OP_COPY_RESIDUAL, g);
      if (g == 0) add_wait(u, LYNX_OP_DECODE_ANCHOR, -1);  // later upgrades follow on the queue
      ops.push_back(u);
    }
  }
  return ops;
}

int check_dims(const Dims& d) {
  size_t a, r, m;
  const int rc = lynx_encoded_sizes(d.B, d.L, d.H, d.D, d.page, d.C, &a, &r, &m);
  if (rc) return rc;
  if (d.ppg < 1) return report_error(LYNX_EINVAL, "pages_per_group must be >= 1");
  return LYNX_OK;
}

int check_ptr16(const void* p) {
  if (!p) return report_error(LYNX_EINVAL, "null pointer");
  if (reinterpret_cast<uintptr_t>(p) & 15u)
    return report_error(LYNX_EINVAL, "pointer not 16-byte aligned");
  return LYNX_OK;
}

int cuda_error(cudaError_t e, const char* what) {
  char msg[200];
  snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
  return report_error(LYNX_ECUDA, msg);
}

// Enqueues a plan.  One event per operation that a later one waits for,
// recorded on the operation's queue right after it; "every group of a kind"
// is the last one of that kind (a kind runs on one in-order queue).
struct Executor {
  const Dims& d;
  cudaStream_t q[3];
  std::vector<lynx_split_op> ops;
  std::vector<cudaEvent_t> ev;   // per op, or null
  std::vector<int64_t> last_of;  // last op index of each kind
  std::vector<std::vector<int64_t>> at;  // [kind][group] -> op index
  explicit Executor(const Dims& dd) : d(dd), q{nullptr, nullptr, nullptr} {}
  ~Executor() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);  // released by the runtime once recorded work completes
  }
  int64_t index_of(int kind, int64_t group) const {
    if (kind < 0 || kind >= (int)at.size()) return -1;
    if (group < 0) return last_of[kind];
    return group < (int64_t)at[kind].size() ? at[kind][group] : -1;
  }
  int prepare() {
    ev.assign(ops.size(), nullptr);
    last_of.assign(6, -1);
    at.assign(6, std::vector<int64_t>((size_t)d.groups(), -1));
    for (size_t i = 0; i < ops.size(); ++i) {
      last_of[ops[i].kind] = (int64_t)i;
      at[ops[i].kind][(size_t)ops[i].group] = (int64_t)i;
    }
    for (size_t i = 0; i < ops.size(); ++i)
      for (int w = 0; w < 2; ++w) {
        if (ops[i].wait_kind[w] == LYNX_OP_NONE) continue;
        const int64_t j = index_of(ops[i].wait_kind[w], ops[i].wait_group[w]);
        if (j < 0 || j >= (int64_t)i) return report_error(LYNX_EINVAL, "malformed schedule");
        if (!ev[j]) {
          cudaError_t e = cudaEventCreateWithFlags(&ev[j], cudaEventDisableTiming);
          if (e != cudaSuccess) return cuda_error(e, "cudaEventCreateWithFlags");
        }
      }
    return LYNX_OK;
  }
  // make op j (if any) record an event when it runs
  int ensure_event(int64_t j) {
    if (j < 0 || ev[j]) return LYNX_OK;
    cudaError_t e = cudaEventCreateWithFlags(&ev[j], cudaEventDisableTiming);
    return e == cudaSuccess ? LYNX_OK : cuda_error(e, "cudaEventCreateWithFlags");
  }
  template <class Run>
  int run(Run&& enqueue) {
    for (size_t i = 0; i < ops.size(); ++i) {
      const lynx_split_op& op = ops[i];
      cudaStream_t s = q[op.queue];
      for (int w = 0; w < 2; ++w) {
        if (op.wait_kind[w] == LYNX_OP_NONE) continue;
        const int64_t j = index_of(op.wait_kind[w], op.wait_group[w]);
        if (ops[j].queue == op.queue) continue;  // same in-order queue
        cudaError_t e = cudaStreamWaitEvent(s, ev[j], 0);
        if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
      }
      const int rc = enqueue(op, s);
      if (rc) return rc;
      if (ev[i]) {
        cudaError_t e = cudaEventRecord(ev[i], s);
        if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
      }
    }
    return LYNX_OK;
  }
  // Record `user` on stream s; with j >= 0, once op j (any queue) is done.
  int signal(cudaEvent_t user, cudaStream_t s, int64_t j) {
    if (!user) return LYNX_OK;
    if (j >= 0) {
      cudaError_t e = cudaStreamWaitEvent(s, ev[j], 0);
      if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
    }
    cudaError_t e = cudaEventRecord(user, s);
    return e == cudaSuccess ? LYNX_OK : cuda_error(e, "cudaEventRecord");
  }
};

}  // namespace
}  // namespace lynx

using namespace lynx;

extern "C" {

int lynx_split_plan(int64_t B, int64_t L, int H_kv, int D, int page, int C,
                    int64_t pages_per_group, int send, int with_decode, lynx_split_op* ops,
                    int64_t max_ops, int64_t* n_ops) {
  Dims d{B, L, H_kv, D, page, C, pages_per_group};
  int rc = check_dims(d);
  if (rc) return rc;
  if (!n_ops) return report_error(LYNX_EINVAL, "null pointer");
  const std::vector<lynx_split_op> plan = build_plan(d, send != 0, with_decode != 0 && !send);
  *n_ops = (int64_t)plan.size();
  if (max_ops < (int64_t)plan.size() || (!ops && !plan.empty()))
    return report_error(LYNX_EWORKSPACE, "ops holds fewer entries than the schedule");
  if (!plan.empty()) memcpy(ops, plan.data(), plan.size() * sizeof(lynx_split_op));
  return LYNX_OK;
}

int lynx_split_receive(const void* h_anchor, const float* h_meta, const void* h_residual,
                       void* anchor, float* meta, void* residual, int64_t B, int64_t L,
                       int H_kv, int D, int page, int C, float alpha, int64_t pages_per_group,
                       void* out, int out_dtype, void* copy_stream, void* hi_stream,
                       void* lo_stream, void* anchor_ready, void* full_ready) {
  Dims d{B, L, H_kv, D, page, C, pages_per_group};
  int rc = check_dims(d);
  if (rc) return rc;
  if (!(alpha > 0.0f) || alpha != alpha || alpha > 3.0e38f)
    return report_error(LYNX_EINVAL, "alpha must be finite and > 0");
  if (out && out_dtype != LYNX_OUT_BF16 && out_dtype != LYNX_OUT_FP32)
    return report_error(LYNX_EINVAL, "out_dtype must be LYNX_OUT_BF16 or LYNX_OUT_FP32");
  Executor x(d);
  x.q[LYNX_Q_COPY] = static_cast<cudaStream_t>(copy_stream);
  x.q[LYNX_Q_HI] = static_cast<cudaStream_t>(hi_stream);
  x.q[LYNX_Q_LO] = static_cast<cudaStream_t>(lo_stream);
  if (d.pages() > 0) {
    for (const void* p : {h_anchor, (const void*)h_meta, h_residual, (const void*)anchor,
                          (const void*)meta, (const void*)residual})
      if ((rc = check_ptr16(p))) return rc;
    if (out && (rc = check_ptr16(out))) return rc;
    x.ops = build_plan(d, false, out != nullptr);
  }
  if ((rc = x.prepare())) return rc;
  // Without out, the phases end with copies: their events let hi / lo record
  // the ready events.  With out, they end with the last kernel of hi / lo.
  const int64_t a_done = out ? -1 : x.last_of[LYNX_OP_COPY_META];
  const int64_t f_done = out ? -1 : x.last_of[LYNX_OP_COPY_RESIDUAL];
  if ((rc = x.ensure_event(a_done)) || (rc = x.ensure_event(f_done))) return rc;
  const size_t osz = out_dtype == LYNX_OUT_FP32 ? 4 : 2;
  rc = x.run([&](const lynx_split_op& op, cudaStream_t s) -> int {
    const size_t o = (size_t)op.offset, n = (size_t)op.bytes;
    cudaError_t e = cudaSuccess;
    switch (op.kind) {
      case LYNX_OP_COPY_ANCHOR:
        e = cudaMemcpyAsync((char*)anchor + o, (const char*)h_anchor + o, n,
                            cudaMemcpyHostToDevice, s);
        break;
      case LYNX_OP_COPY_META:
        e = cudaMemcpyAsync((char*)meta + o, (const char*)h_meta + o, n,
                            cudaMemcpyHostToDevice, s);
        break;
      case LYNX_OP_COPY_RESIDUAL:
        e = cudaMemcpyAsync((char*)residual + o, (const char*)h_residual + o, n,
                            cudaMemcpyHostToDevice, s);
        break;
      case LYNX_OP_DECODE_ANCHOR:
      case LYNX_OP_UPGRADE: {
        const int64_t p0 = op.page0;
        const void* a = (const char*)anchor + p0 * d.anchor_pp();
        const void* r = (const char*)residual + p0 * d.anchor_pp();
        const float* m = (const float*)((const char*)meta + p0 * d.meta_pp());
        void* dst = (char*)out + (size_t)p0 * (size_t)(d.bf16_pp() / 2) * osz;
        const int64_t Lg = op.n_pages * page;
        return op.kind == LYNX_OP_DECODE_ANCHOR
                   ? lynx_decode_anchor(a, m, 1, Lg, H_kv, D, page, C, alpha, dst, out_dtype, s)
                   : lynx_decode_full(a, r, m, 1, Lg, H_kv, D, page, C, alpha, dst, out_dtype,
                                      s);
      }
      default:
        return report_error(LYNX_EINVAL, "unexpected operation in a receive schedule");
    }
    return e == cudaSuccess ? LYNX_OK : cuda_error(e, "cudaMemcpyAsync");
  });
  if (rc) return rc;
  if ((rc = x.signal(static_cast<cudaEvent_t>(anchor_ready), x.q[LYNX_Q_HI], a_done))) return rc;
  return x.signal(static_cast<cudaEvent_t>(full_ready), x.q[LYNX_Q_LO], f_done);
}

int lynx_split_send(const void* kv, int64_t B, int64_t L, int H_kv, int D, int page, int C,
                    float alpha, void* anchor, float* meta, void* residual, void* h_anchor,
                    float* h_meta, void* h_residual, int64_t pages_per_group, void* hi_stream,
                    void* copy_stream, void* anchor_sent, void* all_sent) {
  Dims d{B, L, H_kv, D, page, C, pages_per_group};
  int rc = check_dims(d);
  if (rc) return rc;
  if (!(alpha > 0.0f) || alpha != alpha || alpha > 3.0e38f)
    return report_error(LYNX_EINVAL, "alpha must be finite and > 0");
  Executor x(d);
  x.q[LYNX_Q_COPY] = static_cast<cudaStream_t>(copy_stream);
  x.q[LYNX_Q_HI] = static_cast<cudaStream_t>(hi_stream);
  x.q[LYNX_Q_LO] = static_cast<cudaStream_t>(hi_stream);  // unused by a send schedule
  if (d.pages() > 0) {
    for (const void* p : {kv, (const void*)anchor, (const void*)meta, (const void*)residual,
                          (const void*)h_anchor, (const void*)h_meta, (const void*)h_residual})
      if ((rc = check_ptr16(p))) return rc;
    x.ops = build_plan(d, true, false);
  }
  if ((rc = x.prepare())) return rc;
  const int64_t a_done = x.last_of[LYNX_OP_COPY_META];
  rc = x.run([&](const lynx_split_op& op, cudaStream_t s) -> int {
    const size_t o = (size_t)op.offset, n = (size_t)op.bytes;
    cudaError_t e = cudaSuccess;
    switch (op.kind) {
      case LYNX_OP_ENCODE: {
        const int64_t p0 = op.page0;
        return lynx_encode((const char*)kv + p0 * d.bf16_pp(), 1, op.n_pages * page, H_kv, D,
                           page, C, alpha, (char*)anchor + p0 * d.anchor_pp(),
                           (char*)residual + p0 * d.anchor_pp(),
                           (float*)((char*)meta + p0 * d.meta_pp()), s);
      }
      case LYNX_OP_COPY_ANCHOR:
        e = cudaMemcpyAsync((char*)h_anchor + o, (const char*)anchor + o, n,
                            cudaMemcpyDeviceToHost, s);
        break;
      case LYNX_OP_COPY_META:
        e = cudaMemcpyAsync((char*)h_meta + o, (const char*)meta + o, n,
                            cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess && &op - x.ops.data() == a_done && anchor_sent)
          e = cudaEventRecord(static_cast<cudaEvent_t>(anchor_sent), s);
        break;
      case LYNX_OP_COPY_RESIDUAL:
        e = cudaMemcpyAsync((char*)h_residual + o, (const char*)residual + o, n,
                            cudaMemcpyDeviceToHost, s);
        break;
      default:
        return report_error(LYNX_EINVAL, "unexpected operation in a send schedule");
    }
    return e == cudaSuccess ? LYNX_OK : cuda_error(e, "cudaMemcpyAsync");
  });
  if (rc) return rc;
  if (a_done < 0 && (rc = x.signal(static_cast<cudaEvent_t>(anchor_sent), x.q[LYNX_Q_COPY], -1)))
    return rc;
  return x.signal(static_cast<cudaEvent_t>(all_sent), x.q[LYNX_Q_COPY], -1);
}

// ------------------------------------------------------------ header

// CRC-32 of IEEE 802.3 (reflected polynomial 0xEDB88320, initial and final
// value 0xFFFFFFFF), bit by bit.
static uint32_t crc32_ieee(const unsigned char* p, size_t n) {
  uint32_t c = 0xffffffffu;
  for (size_t i = 0; i < n; ++i) {
    c ^= p[i];
    for (int k = 0; k < 8; ++k) c = (c >> 1) ^ (0xedb88320u & (0u - (c & 1u)));
  }
  return c ^ 0xffffffffu;
}

static const char kMagic[8] = {'L', 'Y', 'N', 'X', 'K', 'V', 0, 1};

static int header_fields(lynx_header* h, int64_t B, int64_t L, int H_kv, int D, int page, int C,
                         float alpha, int with_residual) {
  size_t a, r, m;
  int rc = lynx_encoded_sizes(B, L, H_kv, D, page, C, &a, &r, &m);
  if (rc) return rc;
  if (!(alpha > 0.0f) || alpha != alpha || alpha > 3.0e38f)
    return report_error(LYNX_EINVAL, "alpha must be finite and > 0");
  memset(h, 0, sizeof *h);
  memcpy(h->magic, kMagic, 8);
  h->version = 1;
  h->header_bytes = (uint32_t)sizeof(lynx_header);
  h->B = B;
  h->L = L;
  h->H_kv = H_kv;
  h->D = D;
  h->page = page;
  h->C = C;
  h->alpha = alpha;
  h->flags = with_residual ? 1u : 0u;
  h->anchor_offset = sizeof(lynx_header);
  h->anchor_bytes = a;
  h->meta_offset = h->anchor_offset + a;
  h->meta_bytes = m;
  h->residual_offset = h->meta_offset + m;
  h->residual_bytes = with_residual ? r : 0;
  h->total_bytes = h->residual_offset + h->residual_bytes;
  return LYNX_OK;
}

int lynx_header_init(lynx_header* h, int64_t B, int64_t L, int H_kv, int D, int page, int C,
                     float alpha, int with_residual) {
  if (!h) return report_error(LYNX_EINVAL, "null pointer");
  int rc = header_fields(h, B, L, H_kv, D, page, C, alpha, with_residual);
  if (rc) return rc;
  h->header_crc = crc32_ieee(reinterpret_cast<const unsigned char*>(h), offsetof(lynx_header, header_crc));
  return LYNX_OK;
}

int lynx_header_check(const lynx_header* h) {
  if (!h) return report_error(LYNX_EINVAL, "null pointer");
  if (memcmp(h->magic, kMagic, 8)) return report_error(LYNX_EINVAL, "not a Lynx stream header");
  if (h->version != 1 || h->header_bytes != sizeof(lynx_header))
    return report_error(LYNX_EINVAL, "unsupported header version");
  if (crc32_ieee(reinterpret_cast<const unsigned char*>(h), offsetof(lynx_header, header_crc)) !=
      h->header_crc)
    return report_error(LYNX_EINVAL, "header CRC mismatch");
  if (h->flags & ~1u) return report_error(LYNX_EINVAL, "unknown header flags");
  if (h->reserved[0] | h->reserved[1] | h->reserved[2])
    return report_error(LYNX_EINVAL, "reserved header fields are not zero");
  lynx_header ref;
  int rc = header_fields(&ref, h->B, h->L, h->H_kv, h->D, h->page, h->C, h->alpha,
                         (int)(h->flags & 1u));
  if (rc) return rc;
  ref.header_crc = h->header_crc;
  if (memcmp(&ref, h, sizeof ref))
    return report_error(LYNX_EINVAL, "header sizes or offsets do not follow from its dimensions");
  return LYNX_OK;
}

}  // extern "C"
