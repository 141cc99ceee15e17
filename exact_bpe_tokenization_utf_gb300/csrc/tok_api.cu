// Host side of the C ABI declared in include/tok.h.
//
// A handle owns the device-side vocabulary (merge hash table, per-token
// lengths and operand-length bounds), a workspace that grows to the largest
// input seen and is then reused (no per-call allocation after warm-up), a
// stream, and a pinned status buffer.  A host request costs two host
// synchronisations: one to read the status and id count, one for the ids
// ("TokTier: exact stateful tokenization for agentic LLM serving", Section
// 4.3, cuts a request from eight host syncs to two).
#include <algorithm>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/tok.h"
#include "tok_common.cuh"

using namespace tokgb;

namespace {

constexpr int N_STAGES = 3;
const char* kStageNames[N_STAGES] = {"k_boundaries", "k_bpe_engine", "k_emit"};

thread_local std::string g_load_error;

struct ByteStringHash {
  size_t operator()(const std::string& s) const { return std::hash<std::string>()(s); }
};

}  // namespace

constexpr unsigned long long kDefaultWaitNs = 4000000000ull;  // 4 s

struct tok_handle {
  int dev = 0;
  int n_sms = 1;
  int pattern = 0;
  cudaStream_t stream = nullptr;
  DevVocab v{};
  // device allocations of the vocabulary
  MergeEntry* d_table = nullptr;
  int32_t* d_byte_id = nullptr;
  uint16_t* d_tok_len = nullptr;
  uint16_t* d_max_left = nullptr;
  uint16_t* d_max_right = nullptr;
  WholeEntry* d_whole = nullptr;
  unsigned long long* d_whole_tail = nullptr;
  uint64_t whole_tail_bytes = 0;
  uint32_t* d_pair_bits = nullptr;
  uint32_t n_whole = 0;
  uint64_t hash = 0;
  // workspace
  Workspace ws{};
  int32_t* d_out = nullptr;           // ids of host-side calls
  long long* d_off = nullptr;         // token byte offsets of host-side calls (allocated on first use)
  long long* d_items = nullptr;       // item starts of host-side batch calls
  long long* d_item_off = nullptr;
  uint64_t cap_items = 0;
  DevStatus* h_status = nullptr;      // pinned
  long long* h_ustatus = nullptr;     // pinned, written by the device: code, ids, UTF-8 error offset
  long long* d_ustatus = nullptr;     // its device address
  long long* h_items = nullptr;       // pinned
  uint64_t cap_h_items = 0;
  uint32_t epoch = 0;
  std::string err;
  int64_t err_off = -1;
  uint32_t last_epoch = 0;            // epoch of the latest call
  uint64_t launches = 0;
  bool timing = false;
  cudaEvent_t ev[N_STAGES + 1] = {};
  float stage_ms[N_STAGES] = {};
  bool have_times = false;
  // test hook (tok_debug_fail_alloc): the allocation that fails, counted
  // from 1 = the next one; 0 = none
  uint32_t fail_alloc_in = 0;
  // limit of a device-side wait (the grid barriers of the BPE kernel), and
  // the test hook tok_debug_grid_wait: arrivals a grid barrier waits for
  // beyond the CTAs that come
  unsigned long long wait_ns = kDefaultWaitNs;
  uint32_t grid_extra = 0;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    else prev = -1;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

int fail(tok_handle* h, int code, const std::string& msg) {
  if (h) h->err = msg;
  else g_load_error = msg;
  return code;
}

int cuda_fail(tok_handle* h, cudaError_t e, const char* what) {
  return fail(h, TOK_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

uint64_t fnv1a(uint64_t h, const void* p, size_t n) {
  const uint8_t* b = static_cast<const uint8_t*>(p);
  for (size_t i = 0; i < n; ++i) {
    h ^= b[i];
    h *= 1099511628211ull;
  }
  return h;
}

// group totals held for a workspace of nbch 512-byte chunks
size_t gtot_cap(uint64_t nbch) { return (size_t)(nbch / CTOT_GROUP + 2); }

template <class T>
cudaError_t dalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), std::max<size_t>(count, 1) * sizeof(T));
}

// true when the handle's failure hook says this allocation is the one that
// fails (it then stands in for a cudaMalloc that found the device full)
bool injected_failure(tok_handle* h) {
  return h->fail_alloc_in > 0 && --h->fail_alloc_in == 0;
}

// device allocation of a handle's buffers (workspace, items, offsets)
template <class T>
cudaError_t halloc(tok_handle* h, T** p, size_t count) {
  if (injected_failure(h)) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return dalloc(p, count);
}

// pinned host allocation of a handle's buffers
template <class T>
cudaError_t halloc_pinned(tok_handle* h, T** p, size_t count) {
  if (injected_failure(h)) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMallocHost(reinterpret_cast<void**>(p), std::max<size_t>(count, 1) * sizeof(T));
}

void free_workspace(tok_handle* h) {
  Workspace& w = h->ws;
  // (the group totals live in the status allocation)
  void* ptrs[] = {w.text,     w.pstart,   w.tok,      w.fcnt,     w.sfrag,  w.sbatch,
                  w.wq,       w.longq,    w.st,       w.e_sym[0], w.e_sym[1], w.e_len[0],
                  w.e_len[1], w.e_kr[0],  w.e_kr[1],  w.e_fl,     w.e_rs,   w.edge,
                  h->d_out,   h->d_off};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  w = Workspace{};
  h->d_out = nullptr;
  h->d_off = nullptr;
}

// Grow the workspace to hold n bytes (no-op when it already does).
int ensure_workspace(tok_handle* h, uint64_t n) {
  if (n > MAX_TEXT_BYTES) return fail(h, TOK_EINVAL, "text longer than 2^34 - 2 bytes");
  if (h->ws.st && n <= h->ws.cap_bytes) return TOK_OK;
  uint64_t cap = std::max<uint64_t>(n + n / 4, 1 << 16);
  cap = (cap + CHUNK - 1) / CHUNK * CHUNK;
  free_workspace(h);
  Workspace& w = h->ws;
  const uint64_t nch = cap / CHUNK;
  const uint64_t nbch = cap / BCHUNK;
  const uint64_t pad = 256;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  chk(halloc(h, &w.text, cap + pad));
  chk(halloc(h, &w.pstart, cap / 32 + pad));
  chk(halloc(h, &w.tok, cap + pad));
  // queue sizes: a queued short fragment has >= 2 bytes (a single byte always
  // settles), a warp batch >= 1 short fragment, a wide fragment > SB_MAX
  // bytes, a long one > B_CAP bytes (plus at most one of unknown length per
  // chunk)
  chk(halloc(h, &w.fcnt, cap + pad));
  chk(halloc(h, &w.sfrag, cap / 2 + nbch + pad));
  chk(halloc(h, &w.sbatch, cap / 2 + nbch + pad));
  chk(halloc(h, &w.wq, cap / (SB_MAX + 1) + nbch + pad));
  chk(halloc(h, &w.longq, cap / (B_CAP + 1) + nbch + pad));
  // the status, the group totals, the chunk totals (the group and chunk
  // totals live in the status allocation): the part cleared before a call is
  // one range
  {
    uint8_t* p = nullptr;
    chk(halloc(h, &p, sizeof(DevStatus) + (gtot_cap(nbch) + nbch + 2) * sizeof(uint32_t)));
    w.st = reinterpret_cast<DevStatus*>(p);
    w.gtot = p ? reinterpret_cast<uint32_t*>(p + sizeof(DevStatus)) : nullptr;
    w.ctot = p ? w.gtot + gtot_cap(nbch) : nullptr;
  }
  chk(halloc(h, &w.edge, nch + 2));
  for (int b = 0; b < 2; ++b) {
    chk(halloc(h, &w.e_sym[b], cap + pad));
    chk(halloc(h, &w.e_len[b], cap + pad));
    chk(halloc(h, &w.e_kr[b], cap + pad));
  }
  chk(halloc(h, &w.e_fl, cap + pad));
  chk(halloc(h, &w.e_rs, cap + pad));
  chk(halloc(h, &h->d_out, cap + pad));
  if (e == cudaSuccess) e = cudaMemset(w.pstart, 0, (cap / 32 + pad) * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(w.st, 0, sizeof(DevStatus));
  if (e == cudaSuccess) e = cudaMemset(w.edge, 0, (nch + 2) * sizeof(unsigned long long));
  if (e != cudaSuccess) {
    free_workspace(h);
    cudaGetLastError();
    return fail(h, TOK_ENOMEM, std::string("workspace allocation failed: ") + cudaGetErrorString(e));
  }
  w.cap_bytes = cap;
  w.cap_chunks = nch;
  return TOK_OK;
}

int ensure_items(tok_handle* h, uint64_t n_items) {
  if (n_items + 1 <= h->cap_items && n_items + 1 <= h->cap_h_items) return TOK_OK;
  const uint64_t cap = std::max<uint64_t>(n_items + 1, 64) * 2;
  if (h->d_items) cudaFree(h->d_items);
  if (h->d_item_off) cudaFree(h->d_item_off);
  if (h->h_items) cudaFreeHost(h->h_items);
  h->d_items = nullptr; h->d_item_off = nullptr; h->h_items = nullptr;
  cudaError_t e = halloc(h, &h->d_items, cap);
  if (e == cudaSuccess) e = halloc(h, &h->d_item_off, cap);
  if (e == cudaSuccess) e = halloc_pinned(h, &h->h_items, cap);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (h->d_items) cudaFree(h->d_items);
    if (h->d_item_off) cudaFree(h->d_item_off);
    if (h->h_items) cudaFreeHost(h->h_items);
    h->d_items = nullptr; h->d_item_off = nullptr; h->h_items = nullptr;
    h->cap_items = h->cap_h_items = 0;
    return fail(h, TOK_ENOMEM, "item buffer allocation failed");
  }
  h->cap_items = h->cap_h_items = cap;
  return TOK_OK;
}

// The epoch of a new call.  The UTF-8 error word is keyed by the low 24 bits
// of the epoch (err_key), the chunk-edge words by the whole epoch: when the
// low bits wrap, both are cleared first.
uint32_t next_epoch(tok_handle* h, cudaStream_t s) {
  uint32_t e = ++h->epoch;
  if (e >= 0x3FFFFFFFu) h->epoch = e = 1;
  if ((e & 0xFFFFFFu) <= 1u) {
    cudaMemsetAsync(&h->ws.st->err_off, 0, sizeof(unsigned long long), s);
    cudaMemsetAsync(h->ws.edge, 0, (h->ws.cap_chunks + 2) * sizeof(unsigned long long), s);
  }
  h->last_epoch = e;
  return e;
}

// Clear the status counters, the group totals and the chunk totals of a
// call over n bytes (they follow err_off in one allocation).
void clear_counters(tok_handle* h, uint64_t n, cudaStream_t s) {
  constexpr size_t lo = offsetof(DevStatus, code);
  const size_t nt = gtot_cap(h->ws.cap_bytes / BCHUNK) + (size_t)n_bchunks((long long)n);
  cudaMemsetAsync(reinterpret_cast<uint8_t*>(h->ws.st) + lo, 0, sizeof(DevStatus) - lo + nt * sizeof(uint32_t), s);
}

// Enqueue the whole chain for one call.
int run_chain(tok_handle* h, Call c, cudaStream_t s) {
  c.pf[0] = Prefetch{h->d_whole, (unsigned long long)sizeof(WholeEntry) << h->v.whole_bits};
  c.pf[1] = Prefetch{h->d_whole_tail, h->whole_tail_bytes};
  c.pf[2] = Prefetch{h->d_table, (unsigned long long)sizeof(MergeEntry) << h->v.bits};
  c.pf[3] = Prefetch{h->v.pair_bits, h->v.pair_bits ? 8192ull : 0ull};
  c.pattern = h->pattern;
  c.epoch = next_epoch(h, s);
  if (c.n == 0) {
    launch_status_only(c, h->ws, s);
    h->launches += 1;
    h->have_times = false;
  } else {
    const bool tm = h->timing;
    clear_counters(h, c.n, s);
    c.settle = 1;
    c.wait_ns = h->wait_ns;
    c.grid_extra = h->grid_extra;
    if (tm) cudaEventRecord(h->ev[0], s);
    launch_boundaries(c, h->ws, h->v, s);
    if (tm) cudaEventRecord(h->ev[1], s);
    launch_bpe_engine(c, h->ws, h->v, h->n_sms, s);
    if (tm) cudaEventRecord(h->ev[2], s);
    launch_emit(c, h->ws, h->v, s);
    if (tm) cudaEventRecord(h->ev[3], s);
    h->launches += N_STAGES;
    h->have_times = tm;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  return TOK_OK;
}

void collect_times(tok_handle* h) {
  if (!h->have_times) return;
  for (int k = 0; k < N_STAGES; ++k) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, h->ev[k], h->ev[k + 1]) == cudaSuccess) h->stage_ms[k] = ms;
  }
}

// Read the status after the chain; sync 1 of a host request.
int read_status(tok_handle* h, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(h->h_status, h->ws.st, sizeof(DevStatus), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "status read");
  collect_times(h);
  h->err_off = err_offset(h->last_epoch, h->h_status->err_off);
  if (h->err_off >= 0) {
    char buf[96];
    snprintf(buf, sizeof buf, "invalid UTF-8 at byte %lld", (long long)h->err_off);
    return fail(h, TOK_EUTF8, buf);
  }
  if (h->h_status->code == ST_ETIMEOUT) return fail(h, TOK_ETIMEOUT, "device-side wait gave up");
  if (h->h_status->code != ST_OK) return fail(h, TOK_ECUDA, "device-side internal error");
  return TOK_OK;
}

Call base_call(tok_handle* h, const uint8_t* d_text, uint64_t n) {
  Call c{};
  c.text = d_text;
  c.src = d_text;
  c.n = (long long)n;
  c.item = nullptr;
  c.n_items = 1;
  c.pattern = h->pattern;
  return c;
}

// ---------------------------------------------------------------------------
// Session repair after an append (Section 3.3; Appendix A.2's splice theorem).
// The cut p is the last position inside the old text whose previous code
// point is a letter or a number and whose own code point has another class
// and is not an apostrophe.  Every alternative of the patterns that consumes
// letters or numbers ends at the end of a run of them (or inside it), or
// after a contraction that begins with an apostrophe, so the match covering
// p - 1 ends at p whatever follows; the fragments before p depend on the text
// up to the code point at p, and (no pattern looks behind) the fragments
// from p on only on the text from p on.  So the old tokens before p stay, and
// text[p:] is encoded anew.

namespace hostucd {
#define TOK_UCD_QUAL static const
#include "ucd_table.inc"
#undef TOK_UCD_QUAL
}  // namespace hostucd

uint32_t host_class(uint32_t cp) {
  if (cp < 128u) {
    if ((cp | 32u) - 'a' < 26u) return CLS_L;
    if (cp - '0' < 10u) return CLS_N;
    if (cp == 32u || cp - 9u < 5u) return CLS_W;
    return CLS_O;
  }
  if (cp > 0x10FFFFu) return CLS_O;
  const uint32_t blk = hostucd::tok_ucd_stage1[cp >> 8];
  const uint32_t w = hostucd::tok_ucd_stage2[blk * 16u + ((cp & 255u) >> 4)];
  return (w >> ((cp & 15u) * 2u)) & 3u;
}

// class of the code point that starts at byte k of s[0..n) (its sequence is
// taken as given: the old text of a session has been encoded before)
uint32_t host_class_at(const uint8_t* s, uint64_t n, uint64_t k) {
  const uint32_t b = s[k];
  if (b < 0x80u) return host_class(b);
  int need = b >= 0xF0u ? 3 : b >= 0xE0u ? 2 : b >= 0xC0u ? 1 : 0;
  if (!need || k + (uint64_t)need >= n + 1) return CLS_O;
  uint32_t cp = b & (0x3Fu >> need);
  for (int i = 1; i <= need; ++i) {
    if (k + (uint64_t)i >= n) return CLS_O;
    cp = (cp << 6) | (s[k + i] & 0x3Fu);
  }
  return host_class(cp);
}

// the last certified cut inside old[0..n), or 0; looks back at most `limit` bytes
uint64_t last_cut(const uint8_t* old, uint64_t n, uint64_t limit) {
  if (n == 0) return 0;
  const uint64_t stop = n > limit ? n - limit : 0;
  uint64_t k = n;  // start of the code point after the previous one
  long long cur = -1;
  uint32_t cur_cls = 0;
  while (k > stop) {
    uint64_t j = k - 1;  // start of the code point before k
    while (j > 0 && (old[j] & 0xC0u) == 0x80u && k - j < 4) --j;
    const uint32_t c = host_class_at(old, n, j);
    // (an apostrophe after a word may begin a contraction that the
    // o200k-style pattern attaches to the word, so it is never a cut)
    if (cur >= 0 && (c == CLS_L || c == CLS_N) && cur_cls != c && old[cur] != 0x27u) return (uint64_t)cur;
    cur = (long long)j;
    cur_cls = c;
    k = j;
  }
  return 0;
}

}  // namespace

extern "C" {

int tok_load(const uint8_t* vocab_bytes, const uint64_t* vocab_off, uint32_t n_vocab, const uint32_t* merges,
             uint32_t n_merges, int pattern_id, tok_handle** out) {
  if (!out) return fail(nullptr, TOK_EINVAL, "out is NULL");
  *out = nullptr;
  const bool ignore_merges = (pattern_id & TOK_IGNORE_MERGES) != 0;
  const int pattern = pattern_id & ~TOK_IGNORE_MERGES;
  if (pattern != TOK_PAT_GPT2 && pattern != TOK_PAT_CL100K_STYLE && pattern != TOK_PAT_O200K_STYLE &&
      pattern != TOK_PAT_DEEPSEEK_STYLE)
    return fail(nullptr, TOK_EINVAL, "unknown pattern id");
  if (!vocab_bytes || !vocab_off || (n_merges && !merges)) return fail(nullptr, TOK_EINVAL, "NULL vocabulary");
  if (n_vocab < 256 || n_vocab >= (1u << 20)) return fail(nullptr, TOK_EMERGES, "n_vocab out of range");
  // tokens
  std::unordered_map<std::string, uint32_t, ByteStringHash> index;
  index.reserve(n_vocab * 2);
  std::vector<uint16_t> tok_len(n_vocab);
  for (uint32_t t = 0; t < n_vocab; ++t) {
    if (vocab_off[t + 1] < vocab_off[t]) return fail(nullptr, TOK_EMERGES, "vocab offsets not increasing");
    const uint64_t len = vocab_off[t + 1] - vocab_off[t];
    if (len == 0 || len > 32767) return fail(nullptr, TOK_EMERGES, "token length out of range");
    tok_len[t] = (uint16_t)len;
    std::string s(reinterpret_cast<const char*>(vocab_bytes + vocab_off[t]), len);
    if (!index.emplace(std::move(s), t).second) return fail(nullptr, TOK_EMERGES, "duplicate token bytes");
  }
  std::vector<int32_t> byte_id(256);
  for (int b = 0; b < 256; ++b) {
    auto it = index.find(std::string(1, (char)b));
    if (it == index.end()) return fail(nullptr, TOK_EMERGES, "a single byte has no token");
    byte_id[b] = (int32_t)it->second;
  }
  // merges -> hash table
  uint32_t bits = 10;
  // a quarter full at most: short probe chains for the engines' lookups
  // (a warp waits for its longest)
  while ((1ull << bits) < 4ull * n_merges) ++bits;
  std::vector<MergeEntry> table(1ull << bits, MergeEntry{EMPTY_KEY, 0, 0});
  std::vector<uint16_t> max_left(n_vocab, 0), max_right(n_vocab, 0);
  std::vector<int64_t> last_made(n_vocab, -1), first_used(n_vocab, INT64_MAX);
  const uint32_t mask = (1u << bits) - 1u;
  for (uint32_t r = 0; r < n_merges; ++r) {
    const uint32_t a = merges[2 * r], b = merges[2 * r + 1];
    if (a >= n_vocab || b >= n_vocab) return fail(nullptr, TOK_EMERGES, "merge id out of range");
    std::string s(reinterpret_cast<const char*>(vocab_bytes + vocab_off[a]), tok_len[a]);
    s.append(reinterpret_cast<const char*>(vocab_bytes + vocab_off[b]), tok_len[b]);
    auto it = index.find(s);
    if (it == index.end()) return fail(nullptr, TOK_EMERGES, "merge result not in vocabulary");
    const uint32_t res = it->second;
    const unsigned long long key = ((unsigned long long)a << 32) | b;
    uint32_t slot = merge_slot(key, bits);
    while (table[slot].key != EMPTY_KEY) {
      if (table[slot].key == key) return fail(nullptr, TOK_EMERGES, "duplicate merge pair");
      slot = (slot + 1) & mask;
    }
    table[slot] = MergeEntry{key, r, res};
    max_left[b] = std::max(max_left[b], tok_len[a]);
    max_right[a] = std::max(max_right[a], tok_len[b]);
    last_made[res] = std::max<int64_t>(last_made[res], r);
    first_used[a] = std::min<int64_t>(first_used[a], r);
    first_used[b] = std::min<int64_t>(first_used[b], r);
  }
  // byte pairs held by some merge result: no merge crosses any other pair
  std::vector<uint32_t> pair_bits(2048, 0u);
  {
    std::vector<uint8_t> is_result(n_vocab, 0);
    for (uint32_t i = 0; i <= mask; ++i)
      if (table[i].key != EMPTY_KEY) is_result[table[i].result] = 1;
    for (uint32_t t = 0; t < n_vocab; ++t) {
      if (!is_result[t]) continue;
      const uint8_t* tb = vocab_bytes + vocab_off[t];
      for (uint32_t j = 0; j + 1 < tok_len[t]; ++j) {
        const uint32_t pi = ((uint32_t)tb[j] << 8) | tb[j + 1];
        pair_bits[pi >> 5] |= 1u << (pi & 31);
      }
    }
  }
  bool monotone = true;
  for (uint32_t t = 0; t < n_vocab && monotone; ++t)
    if (last_made[t] >= 0 && first_used[t] != INT64_MAX && first_used[t] <= last_made[t]) monotone = false;

  // Self-encoding tokens: BPE (the textbook rule) of a token's own bytes gives
  // back that token.  A fragment whose bytes equal such a token's encodes to
  // it, which lets the kernels skip the merge loop for it.
  std::unordered_map<unsigned long long, std::pair<uint32_t, uint32_t>> mh;
  mh.reserve(n_merges * 2 + 1);
  for (uint32_t r = 0; r < n_merges; ++r) {
    const unsigned long long key = ((unsigned long long)merges[2 * r] << 32) | merges[2 * r + 1];
    for (uint32_t slot = merge_slot(key, bits);; slot = (slot + 1) & mask)
      if (table[slot].key == key) { mh.emplace(key, std::make_pair(table[slot].rank, table[slot].result)); break; }
  }
  std::vector<uint32_t> whole_tokens;
  uint32_t max_tok_len = 1;
  {
    std::vector<uint32_t> sy;
    for (uint32_t t = 0; t < n_vocab; ++t) {
      const uint32_t len = tok_len[t];
      max_tok_len = std::max(max_tok_len, len);
      if (len < 2) continue;
      sy.assign(len, 0);
      for (uint32_t i = 0; i < len; ++i) sy[i] = (uint32_t)byte_id[vocab_bytes[vocab_off[t] + i]];
      while (sy.size() > 1) {
        uint32_t best = UINT32_MAX, bi = 0, br = 0;
        for (uint32_t i = 0; i + 1 < sy.size(); ++i) {
          auto it = mh.find(((unsigned long long)sy[i] << 32) | sy[i + 1]);
          if (it != mh.end() && it->second.first < best) { best = it->second.first; bi = i; br = it->second.second; }
        }
        if (best == UINT32_MAX) break;
        sy[bi] = br;
        sy.erase(sy.begin() + bi + 1);
      }
      if (ignore_merges || (sy.size() == 1 && sy[0] == t)) whole_tokens.push_back(t);
    }
  }
  uint32_t wbits = 10;
  // a quarter full at most: a miss (most probes) ends after ~1.4 entries on
  // average, and a warp's longest chain is short
  while ((1ull << wbits) < 4ull * whole_tokens.size()) ++wbits;
  std::vector<WholeEntry> whole(1ull << wbits, WholeEntry{0, 0, 0});
  // bytes 8.. of the longer tokens, each from a word boundary, zero-padded
  // to whole 8-byte words (word 0 is never read)
  std::vector<unsigned long long> tail(1, 0ull);
  for (uint32_t t : whole_tokens) {
    const uint32_t len = tok_len[t];
    const uint64_t first = len > 8 ? tail.size() : 0;
    if (len > 255 || first >= (1u << 24)) {
      // without the flag the table only saves work, so a token it cannot
      // hold is encoded by the merge loop instead; with the flag every token
      // must be found
      if (ignore_merges)
        return fail(nullptr, TOK_EMERGES, "ignore_merges needs tokens of at most 255 bytes (and under 128 MiB of them)");
      continue;
    }
    const uint8_t* tb = vocab_bytes + vocab_off[t];
    for (uint32_t i = 8; i < len; i += 8) {
      unsigned long long w = 0;
      for (uint32_t k = 0; k < 8 && i + k < len; ++k) w |= (unsigned long long)tb[i + k] << (8 * k);
      tail.push_back(w);
    }
    const unsigned long long head = bytes_head(tb, len);
    const unsigned long long hv = bytes_hash(head, tb, len);
    uint32_t slot = (uint32_t)(hv >> (64 - wbits));
    while (whole[slot].offlen != 0) slot = (slot + 1) & ((1u << wbits) - 1u);
    whole[slot] = WholeEntry{head, t, ((uint32_t)first << 8) | len};
  }

  tok_handle* h = new tok_handle();
  h->pattern = pattern;
  cudaError_t e = cudaGetDevice(&h->dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sms, cudaDevAttrMultiProcessorCount, h->dev);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = dalloc(&h->d_table, table.size());
  if (e == cudaSuccess) e = dalloc(&h->d_byte_id, 256);
  if (e == cudaSuccess) e = dalloc(&h->d_tok_len, n_vocab);
  if (e == cudaSuccess) e = dalloc(&h->d_max_left, n_vocab);
  if (e == cudaSuccess) e = dalloc(&h->d_max_right, n_vocab);
  if (e == cudaSuccess) e = dalloc(&h->d_whole, whole.size());
  if (e == cudaSuccess) e = dalloc(&h->d_whole_tail, tail.size());
  h->whole_tail_bytes = tail.size() * sizeof(unsigned long long);
  if (e == cudaSuccess) e = dalloc(&h->d_pair_bits, pair_bits.size());
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_pair_bits, pair_bits.data(), pair_bits.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_whole, whole.data(), whole.size() * sizeof(WholeEntry), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_whole_tail, tail.data(), h->whole_tail_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->d_table, table.data(), table.size() * sizeof(MergeEntry), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->d_byte_id, byte_id.data(), 256 * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->d_tok_len, tok_len.data(), n_vocab * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->d_max_left, max_left.data(), n_vocab * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->d_max_right, max_right.data(), n_vocab * 2, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&h->h_status), sizeof(DevStatus));
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&h->h_ustatus), 4 * sizeof(long long));
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->d_ustatus), h->h_ustatus, 0);
  for (int k = 0; k <= N_STAGES && e == cudaSuccess; ++k) e = cudaEventCreate(&h->ev[k]);
  if (e != cudaSuccess) {
    const int code = (e == cudaErrorMemoryAllocation) ? TOK_ENOMEM : TOK_ECUDA;
    std::string msg = std::string("tok_load: ") + cudaGetErrorString(e);
    cudaGetLastError();
    tok_free(h);
    return fail(nullptr, code, msg);
  }
  h->v.table = h->d_table;
  h->v.bits = bits;
  h->v.n_vocab = n_vocab;
  h->v.byte_id = h->d_byte_id;
  h->v.tok_len = h->d_tok_len;
  h->v.max_left = h->d_max_left;
  h->v.max_right = h->d_max_right;
  h->v.monotone = monotone ? 1 : 0;
  h->v.whole = h->d_whole;
  h->v.whole_bits = wbits;
  h->v.max_tok_len = max_tok_len;
  h->v.whole_tail = h->d_whole_tail;
  // with ignore_merges a whole fragment that is any token is that token, so
  // fragments are never split into pieces (a piece may not take that rule)
  h->v.pair_bits = ignore_merges ? nullptr : h->d_pair_bits;
  h->n_whole = (uint32_t)whole_tokens.size();
  uint64_t hh = 1469598103934665603ull;
  hh = fnv1a(hh, &pattern_id, sizeof pattern_id);
  for (uint32_t t = 0; t < n_vocab; ++t) {
    const uint32_t l = tok_len[t];
    hh = fnv1a(hh, &l, sizeof l);
    hh = fnv1a(hh, vocab_bytes + vocab_off[t], l);
  }
  hh = fnv1a(hh, merges, (size_t)n_merges * 2 * sizeof(uint32_t));
  h->hash = hh;
  *out = h;
  return TOK_OK;
}

void tok_free(tok_handle* h) {
  if (!h) return;
  DeviceGuard g(h->dev);
  if (h->stream) cudaStreamSynchronize(h->stream);
  free_workspace(h);
  void* ptrs[] = {h->d_table,  h->d_byte_id,     h->d_tok_len,   h->d_max_left, h->d_max_right, h->d_whole,
                  h->d_whole_tail, h->d_pair_bits, h->d_items, h->d_item_off};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->h_status) cudaFreeHost(h->h_status);
  if (h->h_ustatus) cudaFreeHost(h->h_ustatus);
  if (h->h_items) cudaFreeHost(h->h_items);
  for (int k = 0; k <= N_STAGES; ++k)
    if (h->ev[k]) cudaEventDestroy(h->ev[k]);
  if (h->stream) cudaStreamDestroy(h->stream);
  delete h;
}

const char* tok_last_error(tok_handle* h) { return h ? h->err.c_str() : g_load_error.c_str(); }

int64_t tok_error_offset(tok_handle* h) { return h ? h->err_off : -1; }

uint64_t tok_content_hash(tok_handle* h) { return h ? h->hash : 0; }

uint64_t tok_launch_count(tok_handle* h) { return h ? h->launches : 0; }

int tok_debug_fail_alloc(tok_handle* h, uint32_t k) {
  if (!h) return TOK_EINVAL;
  h->fail_alloc_in = k;
  return TOK_OK;
}

int tok_debug_grid_wait(tok_handle* h, uint32_t extra, uint32_t wait_ms) {
  if (!h) return TOK_EINVAL;
  h->grid_extra = extra;
  h->wait_ns = wait_ms ? (unsigned long long)wait_ms * 1000000ull : kDefaultWaitNs;
  return TOK_OK;
}

int tok_set_timing(tok_handle* h, int enable) {
  if (!h) return TOK_EINVAL;
  h->timing = enable != 0;
  return TOK_OK;
}

int tok_stage_times(tok_handle* h, float* ms, const char** names, int cap) {
  if (!h) return TOK_EINVAL;
  if (!h->have_times) return 0;
  DeviceGuard g(h->dev);
  collect_times(h);
  const int n = std::min(cap, N_STAGES);
  for (int k = 0; k < n; ++k) {
    if (ms) ms[k] = h->stage_ms[k];
    if (names) names[k] = kStageNames[k];
  }
  return n;
}

}  // extern "C"

namespace {

// The device address of a pinned (page-locked, mapped) host buffer, or
// nullptr for any other memory.
void* mapped_device_ptr(const void* p) {
  cudaPointerAttributes a{};
  if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// host in, host out; offsets (or nullptr) receive every token's byte offset
int encode_host(tok_handle* h, const uint8_t* text, uint64_t len, int32_t* ids, int64_t* offsets, uint64_t cap,
                uint64_t* n_ids) {
  if (!h || !n_ids || (len && !text)) return fail(h, TOK_EINVAL, "bad argument");
  DeviceGuard g(h->dev);
  *n_ids = 0;
  int rc = ensure_workspace(h, len);
  if (rc) return rc;
  if (offsets && !h->d_off) {
    const cudaError_t e = halloc(h, &h->d_off, h->ws.cap_bytes + 256);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(h, TOK_ENOMEM, "offset buffer allocation failed");
    }
  }
  cudaStream_t s = h->stream;
  // a pinned input is read by K2 in place (it also fills the device copy the
  // later stages read); any other is copied first
  const uint8_t* src = len ? static_cast<const uint8_t*>(mapped_device_ptr(text)) : nullptr;
  if (len && !src) {
    const cudaError_t e = cudaMemcpyAsync(h->ws.text, text, len, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
  }
  Call c = base_call(h, h->ws.text, len);
  if (src) c.src = src;
  // pinned output buffers large enough for any result: the emit kernel writes
  // the ids (and offsets) and the status straight into host memory, and one
  // synchronisation ends the call
  int32_t* dir_ids = len && cap >= len ? static_cast<int32_t*>(mapped_device_ptr(ids)) : nullptr;
  long long* dir_off = dir_ids && offsets ? static_cast<long long*>(mapped_device_ptr(offsets)) : nullptr;
  if (dir_ids && (!offsets || dir_off)) {
    c.out = dir_ids;
    c.out_off = dir_off;
    c.out_host = 1;
    c.user_status = h->d_ustatus;
    rc = run_chain(h, c, s);
    if (rc) return rc;
    const cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "encode");
    collect_times(h);
    const long long code = h->h_ustatus[0];
    h->err_off = h->h_ustatus[2];
    if (code == TOK_EUTF8) {
      char buf[96];
      snprintf(buf, sizeof buf, "invalid UTF-8 at byte %lld", (long long)h->err_off);
      return fail(h, TOK_EUTF8, buf);
    }
    if (code == ST_ETIMEOUT) return fail(h, TOK_ETIMEOUT, "device-side wait gave up");
    if (code != ST_OK) return fail(h, TOK_ECUDA, "device-side internal error");
    *n_ids = (uint64_t)h->h_ustatus[1];
    return TOK_OK;
  }
  c.out = h->d_out;
  c.out_off = offsets ? h->d_off : nullptr;
  rc = run_chain(h, c, s);
  if (rc) return rc;
  rc = read_status(h, s);
  if (rc) return rc;
  const uint64_t n = h->h_status->n_ids;
  *n_ids = n;
  if (n > cap) return fail(h, TOK_EBUF, "output buffer too small");
  if (n) {
    if (!ids) return fail(h, TOK_EINVAL, "ids is NULL");
    cudaError_t e = cudaMemcpyAsync(ids, h->d_out, n * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && offsets)
      e = cudaMemcpyAsync(offsets, h->d_off, n * sizeof(int64_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "id copy");
  }
  return TOK_OK;
}

}  // namespace

extern "C" {

int tok_encode(tok_handle* h, const uint8_t* text, uint64_t len, int32_t* ids, uint64_t cap, uint64_t* n_ids) {
  return encode_host(h, text, len, ids, nullptr, cap, n_ids);
}

int tok_encode_offsets(tok_handle* h, const uint8_t* text, uint64_t len, int32_t* ids, int64_t* offsets,
                       uint64_t cap, uint64_t* n_ids) {
  if (!offsets) return fail(h, TOK_EINVAL, "offsets is NULL");
  return encode_host(h, text, len, ids, offsets, cap, n_ids);
}

int tok_repair_append(tok_handle* h, const uint8_t* text, uint64_t old_len, uint64_t len, const int32_t* old_ids,
                      const int64_t* old_offsets, uint64_t old_n, int32_t* ids, int64_t* offsets, uint64_t cap,
                      uint64_t* n_ids, uint64_t* reencoded) {
  if (!h || !n_ids || !ids || !offsets || (len && !text) || old_len > len || (old_n && (!old_ids || !old_offsets)))
    return fail(h, TOK_EINVAL, "bad argument");
  *n_ids = 0;
  if (reencoded) *reencoded = 0;
  const uint64_t p = last_cut(text, old_len, 1ull << 20);
  // the old tokens before the cut; the cut must be a token start of them
  const uint64_t k = (uint64_t)(std::lower_bound(old_offsets, old_offsets + old_n, (int64_t)p) - old_offsets);
  if (p && (k >= old_n || (uint64_t)old_offsets[k] != p))
    return fail(h, TOK_EINVAL, "the old token offsets do not belong to this text");
  if (k > cap) {
    // the kept tokens alone overflow: the required size still counts the
    // tail's tokens (encoded with no room, which reports their number)
    uint64_t m = 0;
    const int rc = encode_host(h, text + p, len - p, nullptr, nullptr, 0, &m);
    if (rc != TOK_OK && rc != TOK_EBUF) return rc;
    *n_ids = k + m;
    return fail(h, TOK_EBUF, "output buffer too small");
  }
  if (ids != old_ids) std::copy(old_ids, old_ids + k, ids);
  if (offsets != old_offsets) std::copy(old_offsets, old_offsets + k, offsets);
  uint64_t m = 0;
  const int rc = encode_host(h, text + p, len - p, ids + k, offsets + k, cap - k, &m);
  if (rc == TOK_EBUF) *n_ids = k + m;
  if (rc) {
    if (rc == TOK_EUTF8) h->err_off += (int64_t)p;
    return rc;
  }
  for (uint64_t i = 0; i < m; ++i) offsets[k + i] += (int64_t)p;
  *n_ids = k + m;
  if (reencoded) *reencoded = len - p;
  return TOK_OK;
}

int tok_encode_batch(tok_handle* h, const uint8_t* const* texts, const uint64_t* lens, uint32_t n, int32_t* ids,
                     uint64_t cap, uint64_t* item_off) {
  if (!h || (n && (!texts || !lens)) || !item_off) return fail(h, TOK_EINVAL, "bad argument");
  DeviceGuard g(h->dev);
  uint64_t total = 0;
  for (uint32_t k = 0; k < n; ++k) {
    if (lens[k] && !texts[k]) return fail(h, TOK_EINVAL, "NULL item");
    total += lens[k];
  }
  int rc = ensure_workspace(h, total);
  if (rc) return rc;
  rc = ensure_items(h, n);
  if (rc) return rc;
  cudaStream_t s = h->stream;
  uint64_t pos = 0;
  for (uint32_t k = 0; k < n; ++k) {
    h->h_items[k] = (long long)pos;
    if (lens[k]) {
      const cudaError_t e = cudaMemcpyAsync(h->ws.text + pos, texts[k], lens[k], cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
    }
    pos += lens[k];
  }
  h->h_items[n] = (long long)total;
  cudaError_t e = cudaMemcpyAsync(h->d_items, h->h_items, (n + 1) * sizeof(long long), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "item copy");
  Call c = base_call(h, h->ws.text, total);
  c.item = h->d_items;
  c.n_items = (int)n;
  c.out = h->d_out;
  c.item_off = h->d_item_off;
  rc = run_chain(h, c, s);
  if (rc) return rc;
  rc = read_status(h, s);
  if (rc) return rc;
  const uint64_t nid = h->h_status->n_ids;
  if (nid > cap) {
    item_off[n] = nid;
    return fail(h, TOK_EBUF, "output buffer too small");
  }
  if (nid && !ids) return fail(h, TOK_EINVAL, "ids is NULL");
  if (nid) e = cudaMemcpyAsync(ids, h->d_out, nid * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->h_items, h->d_item_off, (n + 1) * sizeof(long long),
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "id copy");
  for (uint32_t k = 0; k <= n; ++k) item_off[k] = (uint64_t)h->h_items[k];
  return TOK_OK;
}

int tok_encode_device(tok_handle* h, const uint8_t* d_text, uint64_t len, int32_t* d_ids, uint64_t cap,
                      int64_t* d_status, void* stream) {
  return tok_encode_offsets_device(h, d_text, len, d_ids, nullptr, cap, d_status, stream);
}

int tok_encode_offsets_device(tok_handle* h, const uint8_t* d_text, uint64_t len, int32_t* d_ids,
                              int64_t* d_offsets, uint64_t cap, int64_t* d_status, void* stream) {
  if (!h || !d_status || (len && (!d_text || !d_ids))) return fail(h, TOK_EINVAL, "bad argument");
  if (cap < len) return fail(h, TOK_EBUF, "cap must be >= len");
  DeviceGuard g(h->dev);
  int rc = ensure_workspace(h, len);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);  // NULL: the CUDA default stream
  Call c = base_call(h, d_text, len);
  c.out = d_ids;
  c.out_off = reinterpret_cast<long long*>(d_offsets);
  c.user_status = reinterpret_cast<long long*>(d_status);
  return run_chain(h, c, s);
}

int tok_encode_batch_device(tok_handle* h, const uint8_t* d_text, uint64_t len, const int64_t* d_item_start,
                            uint32_t n, int32_t* d_ids, uint64_t cap, int64_t* d_item_off, int64_t* d_status,
                            void* stream) {
  if (!h || !d_status || !d_item_start || !d_item_off || n == 0 || (len && (!d_text || !d_ids)))
    return fail(h, TOK_EINVAL, "bad argument");
  if (cap < len) return fail(h, TOK_EBUF, "cap must be >= len");
  DeviceGuard g(h->dev);
  int rc = ensure_workspace(h, len);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);  // NULL: the CUDA default stream
  Call c = base_call(h, d_text, len);
  c.item = reinterpret_cast<const long long*>(d_item_start);
  c.n_items = (int)n;
  c.out = d_ids;
  c.item_off = reinterpret_cast<long long*>(d_item_off);
  c.user_status = reinterpret_cast<long long*>(d_status);
  return run_chain(h, c, s);
}

// Pre-tokenizer only, over items packed back to back (items == nullptr: one
// item).  Fragment starts are offsets into the concatenation.
static int pretokenize_impl(tok_handle* h, uint64_t len, uint32_t n_items, bool batch, int64_t* starts,
                            uint64_t cap, uint64_t* n) {
  cudaStream_t s = h->stream;
  Call c = base_call(h, h->ws.text, len);
  if (batch) {
    c.item = h->d_items;
    c.n_items = (int)n_items;
  }
  c.pattern = h->pattern;
  c.epoch = next_epoch(h, s);
  clear_counters(h, 0, s);
  launch_boundaries(c, h->ws, DevVocab{}, s);
  h->launches += 1;
  h->have_times = false;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  int rc = read_status(h, s);
  if (rc) return rc;
  const uint64_t nw = (len + 31) / 32;
  std::vector<uint32_t> bits(nw);
  e = cudaMemcpy(bits.data(), h->ws.pstart, nw * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "bitmask copy");
  uint64_t cnt = 0;
  for (uint64_t w = 0; w < nw; ++w) {
    uint32_t v = bits[w];
    while (v) {
      const int b = __builtin_ctz(v);
      v &= v - 1;
      const uint64_t p = w * 32 + (uint64_t)b;
      if (p >= len) break;
      if (cnt < cap && starts) starts[cnt] = (int64_t)p;
      ++cnt;
    }
  }
  *n = cnt;
  if (cnt > cap) return fail(h, TOK_EBUF, "starts buffer too small");
  return TOK_OK;
}

int tok_pretokenize(tok_handle* h, const uint8_t* text, uint64_t len, int64_t* starts, uint64_t cap, uint64_t* n) {
  if (!h || !n || (len && !text)) return fail(h, TOK_EINVAL, "bad argument");
  DeviceGuard g(h->dev);
  *n = 0;
  int rc = ensure_workspace(h, len);
  if (rc) return rc;
  if (len == 0) return TOK_OK;
  const cudaError_t e = cudaMemcpyAsync(h->ws.text, text, len, cudaMemcpyHostToDevice, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
  return pretokenize_impl(h, len, 1, false, starts, cap, n);
}

int tok_pretokenize_batch(tok_handle* h, const uint8_t* const* texts, const uint64_t* lens, uint32_t n_items,
                          int64_t* starts, uint64_t cap, uint64_t* n) {
  if (!h || !n || (n_items && (!texts || !lens))) return fail(h, TOK_EINVAL, "bad argument");
  DeviceGuard g(h->dev);
  *n = 0;
  uint64_t total = 0;
  for (uint32_t k = 0; k < n_items; ++k) total += lens[k];
  int rc = ensure_workspace(h, total);
  if (rc) return rc;
  rc = ensure_items(h, n_items);
  if (rc) return rc;
  if (total == 0) return TOK_OK;
  cudaStream_t s = h->stream;
  uint64_t pos = 0;
  for (uint32_t k = 0; k < n_items; ++k) {
    h->h_items[k] = (long long)pos;
    if (lens[k]) {
      const cudaError_t e = cudaMemcpyAsync(h->ws.text + pos, texts[k], lens[k], cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "input copy");
    }
    pos += lens[k];
  }
  h->h_items[n_items] = (long long)total;
  const cudaError_t e =
      cudaMemcpyAsync(h->d_items, h->h_items, (n_items + 1) * sizeof(long long), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "item copy");
  return pretokenize_impl(h, total, n_items, true, starts, cap, n);
}

}  // extern "C"
