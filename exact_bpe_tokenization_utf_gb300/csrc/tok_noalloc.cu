// tok_pretokenize_device_noalloc: the pre-tokenizer for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside another
// framework's memory pool or arena (where a stray cudaMalloc fragments or
// breaks the pool's accounting), code that must not synchronise the device
// (cudaMalloc/cudaFree can serialise with in-flight work), and hosts that run
// with a fixed, pre-reserved memory budget.  This entry point takes device
// input and output buffers from the caller and keeps the only scratch it
// needs (the status block the boundary kernel writes) in a file-scope
// __device__ array of fixed size, which every GPU that loads the library
// holds until the process exits.
#include "../../include/tok.h"
#include "tok_common.cuh"

using namespace tokgb;

namespace {

struct NoAllocScratch {
  DevStatus st;
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

// The device address of g_noalloc_scratch is looked up once per device with
// cudaGetSymbolAddress; each device also counts its calls (the epoch keys the
// UTF-8 error word, see err_key).
constexpr int kMaxDevices = 64;
NoAllocScratch* g_scratch_addr[kMaxDevices] = {};
uint32_t g_epoch[kMaxDevices] = {};

__global__ void k_noalloc_status(const NoAllocScratch* s, uint32_t epoch, long long* d_status) {
  const long long eo = err_offset(epoch, s->st.err_off);
  d_status[0] = eo >= 0 ? TOK_EUTF8 : TOK_OK;
  d_status[1] = eo;
}

// empty text: nothing to split, nothing malformed
__global__ void k_noalloc_empty(long long* d_status) {
  d_status[0] = TOK_OK;
  d_status[1] = -1;
}

}  // namespace

extern "C" int tok_pretokenize_device_noalloc(int pattern_id, const uint8_t* d_text, uint64_t len,
                                              uint32_t* d_start_bits, int64_t* d_status, void* stream) {
  if (pattern_id != TOK_PAT_GPT2 && pattern_id != TOK_PAT_CL100K_STYLE && pattern_id != TOK_PAT_O200K_STYLE &&
      pattern_id != TOK_PAT_DEEPSEEK_STYLE)
    return TOK_EINVAL;
  if (!d_status || (len && (!d_text || !d_start_bits))) return TOK_EINVAL;
  // the same bound as every other entry point: the chunk grid and the UTF-8
  // error word hold positions below 2^34; checked before any device call
  if (len > MAX_TEXT_BYTES) return TOK_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TOK_ECUDA;
  if (!g_scratch_addr[dev]) {
    // once per device, with that device current; the first call on a device
    // should therefore come before any stream capture
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return TOK_ECUDA;
    }
    g_scratch_addr[dev] = static_cast<NoAllocScratch*>(p);
  }
  NoAllocScratch* scratch = g_scratch_addr[dev];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t epoch = ++g_epoch[dev];
  if (epoch >= 0x3FFFFFFFu) g_epoch[dev] = epoch = 1;
  if ((epoch & 0xFFFFFFu) <= 1u &&
      cudaMemsetAsync(&scratch->st.err_off, 0, sizeof(unsigned long long), s) != cudaSuccess) {
    cudaGetLastError();
    return TOK_ECUDA;
  }
  Workspace w{};
  w.st = &scratch->st;
  w.pstart = d_start_bits;
  Call c{};
  c.text = d_text;
  c.src = d_text;
  c.n = (long long)len;
  c.item = nullptr;
  c.n_items = 1;
  c.pattern = pattern_id;
  c.epoch = epoch;
  if (len) {
    launch_boundaries(c, w, DevVocab{}, s);
    k_noalloc_status<<<1, 1, 0, s>>>(scratch, epoch, reinterpret_cast<long long*>(d_status));
  } else {
    k_noalloc_empty<<<1, 1, 0, s>>>(reinterpret_cast<long long*>(d_status));
  }
  return cudaGetLastError() == cudaSuccess ? TOK_OK : TOK_ECUDA;
}
