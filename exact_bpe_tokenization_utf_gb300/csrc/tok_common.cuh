// Shared definitions of the GB300 exact BPE tokenizer library.
//
// Pipeline (one pass over a text or a packed batch; "TokTier: exact stateful
// tokenization for agentic LLM serving", Section 4):
//   K2 boundaries    per 1 KiB chunk: UTF-8 validation + per-code-point class +
//                    run decomposition rules -> fragment-start bitmask
//                    (Section 4.1); the run states at the chunk's edges come
//                    from its halo (or the text beyond).  In encode calls K2 then
//                    settles every fragment that is one byte, or whose bytes
//                    are a token that encodes to itself, with one probe, and
//                    queues the others: those of at most 32 bytes packed into
//                    warp batches, 33..B_CAP bytes one by one, longer ones
//                    (Section 4.2).  A fragment across a chunk edge is handled
//                    by the second of the edge's two CTAs to get there.
//   K3b bpe_engine   persistent: CTAs take fragments longer than B_CAP bytes
//                    (arrays in global memory), then 33..B_CAP-byte fragments
//                    (shared memory; sweeps that merge all certified-safe
//                    pairs), then warps take short batches (one symbol per
//                    lane): batches of fragments of at most 16 bytes merge
//                    each fragment's leftmost lowest-rank pair per step, the
//                    others run certified sweeps.  Every fragment's id count
//                    is added to the total of its 512-byte chunk and of that
//                    chunk's group.
//   K5 emit          per chunk: ids before it (group totals, then chunk
//                    totals), fragment counts -> offsets, copy of the ids in
//                    text order
// Every stage leaves a fragment's ids at the fragment's byte offset in `tok`
// and their number at the same offset in `fcnt`.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace tokgb {

constexpr int CHUNK = 1024;        // bytes per chunk (every per-chunk kernel)
constexpr int CHUNK_THREADS = 128; // 8 bytes per thread in K2
constexpr int BYTES_PER_THREAD = CHUNK / CHUNK_THREADS;
constexpr int HALO = 16;           // look-behind / look-ahead bytes around a chunk
constexpr int BCHUNK = 512;        // bytes per chunk total and per emit CTA (K5)
constexpr int B_THREADS = 128;     // K3b, K5
constexpr int B_CAP = 256;         // longest fragment of the K3b shared-memory engine; longer ones use global memory
constexpr int B_EPT = B_CAP / B_THREADS; // engine symbols per thread at most
constexpr int SB_MAX = 32;         // bytes (symbols) of a warp batch
constexpr unsigned long long MAX_TEXT_BYTES = (1ull << 34) - 2;  // chunk-edge words hold positions + 1 in 34 bits
constexpr int CTOT_GROUP = 64;     // chunks per group total (K5 sums group totals, then chunk totals)
constexpr uint32_t NO_RANK = 0xFFFFFFFFu;
constexpr unsigned long long EMPTY_KEY = ~0ull;

// code point classes of the pre-tokenizer patterns
enum : uint32_t { CLS_O = 0, CLS_L = 1, CLS_N = 2, CLS_W = 3 };

// status codes mirrored from tok.h
enum : int32_t { ST_OK = 0, ST_EUTF8 = -2, ST_EBUF = -5, ST_ETIMEOUT = -6, ST_EINTERNAL = -4 };

// merge table entry: key = left << 32 | right; rank = merge index; result id
struct __align__(16) MergeEntry {
  unsigned long long key;
  uint32_t rank;
  uint32_t result;
};

// whole-token table entry: a token whose own bytes encode to itself, keyed by
// a hash of those bytes.  Its first 8 bytes are in the entry, so that a probe
// of a fragment of at most 8 bytes needs no second load; the rest of a longer
// token is in the tail array, as whole 8-byte words (zero above the end), so
// that its compare takes one load per 8 bytes.  offlen == 0 marks an empty
// slot (len is 2..255).
struct __align__(16) WholeEntry {
  unsigned long long head;  // first min(len, 8) bytes, little-endian, zero above
  uint32_t token;
  uint32_t offlen;          // first tail word (tokens of more than 8 bytes) << 8 | len
};

struct DevVocab {
  const MergeEntry* table;
  uint32_t bits;              // log2(capacity)
  uint32_t n_vocab;
  const WholeEntry* whole;    // tokens t with BPE(bytes(t)) == [t], length >= 2
  uint32_t whole_bits;        // log2(capacity)
  uint32_t max_tok_len;
  const unsigned long long* whole_tail;  // bytes 8.. of the whole-table tokens longer than 8 bytes
  const int32_t* byte_id;     // 256 entries: initial symbol of each byte value
  const uint16_t* tok_len;    // byte length of every token
  const uint16_t* max_left;   // longest left operand of any merge whose right operand is t
  const uint16_t* max_right;  // longest right operand of any merge whose left operand is t
  int monotone;               // every merge that uses a token comes after every merge making it
  // 65,536 bits: bit (x << 8 | y) is set when some merge result's bytes hold
  // the byte pair x y; no merge joins two symbols across a pair whose bit is
  // clear (the result would hold it), so a fragment splits there into
  // pieces that encode independently
  const uint32_t* pair_bits;
};

// a queued fragment: its first byte and its length (-1: ends at the next
// fragment start, to be found)
struct Frag {
  long long start;
  long long len;
};

// device-side per-call status and work counters
struct DevStatus {
  // kept across calls
  unsigned long long err_off;   // first malformed UTF-8 byte of the latest call that had one: err_key
  // cleared before every call, together with the group totals that follow
  // the status in its allocation (one memset)
  int32_t code;
  uint32_t pad0;
  unsigned long long n_ids;
  unsigned long long sfrag_count;  // short fragments queued
  uint32_t sbatch_count;           // warp batches of short fragments
  uint32_t wide_count;             // fragments of 33..B_CAP bytes
  uint32_t long_count, long_taken; // longer fragments
  // warp batches claimed by K3b's warps beyond their first one: many warps
  // add to it while the grid engine waits at its barriers, so each has a
  // line of its own
  alignas(128) uint32_t sbatch_taken;
  // the grid engine of K3b: its barrier (arrivals, generation), the flag a
  // CTA sets when it gave up waiting, and per sweep whether a pair merges
  alignas(128) uint32_t gb_count;
  uint32_t gb_gen, g_abort, g_any[3];
};
static_assert(sizeof(DevStatus) % 16 == 0, "the group totals follow the status");

struct Workspace {
  uint8_t* text;            // device copy of host input (host entry points)
  uint32_t* pstart;         // fragment-start bitmask
  int32_t* tok;             // a fragment's ids, at the fragment's byte offset
  int32_t* fcnt;            // a fragment's number of ids, at its byte offset
  unsigned long long* sfrag;   // short fragments: start << 8 | length, in batch order
  unsigned long long* sbatch;  // warp batches: first sfrag index << 5 | (fragments - 1)
  Frag* wq;                 // fragments of 33..B_CAP bytes
  Frag* longq;              // longer fragments (K3b, global-memory engine)
  unsigned long long* edge; // per 1 KiB chunk edge: edge_word of the first CTA there (k_boundaries)
  uint32_t* ctot;           // ids of the fragments that start in each 512-byte chunk (added up as they finish)
  uint32_t* gtot;           // the same for each group of CTOT_GROUP chunks
  DevStatus* st;
  // global-memory engine storage, indexed by byte position of the fragment
  uint32_t* e_sym[2];
  uint16_t* e_len[2];
  unsigned long long* e_kr[2];
  uint8_t* e_fl;
  int32_t* e_rs;
  uint64_t cap_bytes;       // capacity in bytes of the per-byte arrays
  uint64_t cap_chunks;
};

// a device range K2 prefetches into L2 (the vocabulary tables the probes
// and the BPE engine read)
struct Prefetch {
  const void* p;
  unsigned long long bytes;
};

struct Call {
  const uint8_t* text;        // device: the text the BPE stages and the emit read
  const uint8_t* src;         // where K2 reads the text: `text` itself, or a pinned host buffer's
                              // device address, from which K2 also fills `text` (its own chunk)
  long long n;                // bytes
  const long long* item;      // device item starts, n_items + 1 entries
  int n_items;
  int pattern;
  uint32_t epoch;
  int32_t* out;               // device ids
  long long* out_off;         // device: byte offset of every id's token (nullptr: not wanted)
  long long* item_off;        // device, n_items + 1 (batch) or nullptr
  long long* user_status;     // device int64[4] or nullptr
  int settle;                 // K2 also settles fragments and fills the queues (encode calls)
  int out_host;               // `out` is pinned host memory (mapped): K5 stages a chunk's ids for coalesced stores
  int grid_ctas;              // K3b CTAs that run the grid engine (0: none)
  uint32_t grid_extra;        // arrivals a grid barrier waits for beyond grid_ctas (0; a test sets 1)
  unsigned long long wait_ns; // limit of a device-side wait, in ns of the global timer
  Prefetch pf[4];             // whole-token table, its tail words, merge table, byte-pair bits
};

// The first malformed UTF-8 byte of a call, as one word that atomicMax keeps
// across calls without a reset: the call's epoch (24 bits) above the
// complement of the offset (40 bits).  A later call's key is larger (until
// the epoch wraps, when the host clears the word); within a call the smallest
// offset gives the largest key.
constexpr unsigned long long ERR_OFF_MASK = (1ull << 40) - 1ull;
__host__ __device__ inline unsigned long long err_key(uint32_t epoch, unsigned long long off) {
  return ((unsigned long long)(epoch & 0xFFFFFFu) << 40) | (ERR_OFF_MASK - off);
}
// the offset in a key written by the call with this epoch, or -1
__host__ __device__ inline long long err_offset(uint32_t epoch, unsigned long long key) {
  if ((key >> 40) != (epoch & 0xFFFFFFu) || (key & ERR_OFF_MASK) == 0) return -1;
  return (long long)(ERR_OFF_MASK - (key & ERR_OFF_MASK));
}

__host__ __device__ inline uint32_t merge_slot(unsigned long long key, uint32_t bits) {
  return (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> (64 - bits));
}

// first min(len, 8) bytes of s, little-endian, zero above
__host__ __device__ inline unsigned long long bytes_head(const uint8_t* s, int len) {
  unsigned long long v = 0;
  for (int i = 0; i < len && i < 8; ++i) v |= (unsigned long long)s[i] << (8 * i);
  return v;
}

// 64-bit hash of a byte string from its head (bytes_head), its length and
// the bytes after the first 8 (FNV-1a steps, then the splitmix64 finaliser)
__host__ __device__ inline unsigned long long bytes_hash(unsigned long long head, const uint8_t* s, int len) {
  unsigned long long h = head ^ (0x9E3779B97F4A7C15ull * (unsigned long long)len);
  for (int i = 8; i < len; ++i) {
    h ^= s[i];
    h *= 1099511628211ull;
  }
  h ^= h >> 30;
  h *= 0xBF58476D1CE4E5B9ull;
  h ^= h >> 27;
  h *= 0x94D049BB133111EBull;
  h ^= h >> 31;
  return h;
}

#ifdef __CUDACC__
// Probe the merge table for (a, b): returns (rank << 32 | result), or ~0 when
// the pair is not a merge.  Linear probing over a table at most half full,
// so an empty slot always ends the probe; the loop is bounded anyway.
__device__ __forceinline__ unsigned long long merge_lookup(const DevVocab& v, uint32_t a, uint32_t b) {
  const unsigned long long key = ((unsigned long long)a << 32) | b;
  const uint32_t mask = (1u << v.bits) - 1u;
  uint32_t s = merge_slot(key, v.bits);
  for (uint32_t probe = 0; probe <= mask; ++probe) {
    const uint4 e = __ldg(reinterpret_cast<const uint4*>(v.table + s));
    const unsigned long long k = ((unsigned long long)e.y << 32) | e.x;
    if (k == key) return ((unsigned long long)e.z << 32) | e.w;
    if (k == EMPTY_KEY) break;
    s = (s + 1u) & mask;
  }
  return ~0ull;
}

// Token whose bytes equal s[0..len) and whose own bytes encode to itself,
// or -1.  The hash only selects the first slot; the length and the first 8
// bytes are compared in the entry, the rest against the token's tail words.  Split
// in parts so that a thread can issue the first probes of several strings
// before it waits for any: whole_first_slot gives the first slot of a hash,
// whole_lookup_at finishes from the loaded first entry.
__device__ __forceinline__ bool whole_eligible(const DevVocab& v, int len) {
  return len >= 2 && len <= 255 && len <= (int)v.max_tok_len;
}

__device__ __forceinline__ uint32_t whole_first_slot(const DevVocab& v, unsigned long long h) {
  return (uint32_t)(h >> (64 - v.whole_bits));
}

// First min(len, 8) bytes at p, little-endian, zero above: three aligned
// 32-bit loads and two funnel shifts.  The 12 bytes from p rounded down to a
// multiple of 4 must be readable (shared-memory buffers with room after the
// string).
__device__ __forceinline__ unsigned long long head8(const uint8_t* p, int len) {
  const uintptr_t u = reinterpret_cast<uintptr_t>(p);
  const uint32_t* q = reinterpret_cast<const uint32_t*>(u & ~uintptr_t(3));
  const uint32_t sh = (uint32_t)(u & 3u) * 8u;
  const uint32_t w0 = q[0], w1 = q[1], w2 = q[2];
  unsigned long long v = ((unsigned long long)__funnelshift_r(w1, w2, sh) << 32) | __funnelshift_r(w0, w1, sh);
  if (len < 8) v &= (1ull << (8 * len)) - 1ull;
  return v;
}

// `s` is read with head8: len + 11 bytes from s (rounded down to 4) must be
// readable.
__device__ __forceinline__ int whole_lookup_at(const DevVocab& v, const uint8_t* s, int len,
                                               unsigned long long head, uint32_t slot, uint4 e) {
  const uint32_t mask = (1u << v.whole_bits) - 1u;
  for (uint32_t probe = 0; probe <= mask; ++probe) {
    if (probe) e = __ldg(reinterpret_cast<const uint4*>(v.whole + slot));
    if (e.w == 0u) return -1;
    if ((e.w & 255u) == (uint32_t)len && (((unsigned long long)e.y << 32) | e.x) == head) {
      // bytes 8.. against the tail words (most longer tokens have one)
      const unsigned long long* t = v.whole_tail + (e.w >> 8);
      bool eq = true;
#pragma unroll 1
      for (int i = 8; i < len; i += 8) eq &= __ldg(t++) == head8(s + i, len - i);
      if (eq) return (int)e.z;
    }
    slot = (slot + 1u) & mask;
  }
  return -1;
}

// Record a device-side error of the call; the first error stays.
__device__ __forceinline__ void set_error(DevStatus* st, int32_t code) { atomicCAS(&st->code, (int32_t)ST_OK, code); }

__device__ __forceinline__ uint32_t kr_rank(unsigned long long kr) { return (uint32_t)(kr >> 32); }
__device__ __forceinline__ uint32_t kr_result(unsigned long long kr) { return (uint32_t)kr; }

// Strict UTF-8 (RFC 3629, Section 4): length of the well-formed sequence at
// s[0..avail), or 0 if it is malformed or truncated.  *cp receives the value.
__device__ __forceinline__ int utf8_decode(const uint8_t* s, int avail, uint32_t* cp) {
  const uint32_t b0 = s[0];
  if (b0 < 0x80u) { *cp = b0; return 1; }
  int need;
  uint32_t lo = 0x80u, hi = 0xBFu;
  if (b0 >= 0xC2u && b0 <= 0xDFu) need = 1;
  else if (b0 == 0xE0u) { need = 2; lo = 0xA0u; }
  else if ((b0 >= 0xE1u && b0 <= 0xECu) || b0 == 0xEEu || b0 == 0xEFu) need = 2;
  else if (b0 == 0xEDu) { need = 2; hi = 0x9Fu; }
  else if (b0 == 0xF0u) { need = 3; lo = 0x90u; }
  else if (b0 >= 0xF1u && b0 <= 0xF3u) need = 3;
  else if (b0 == 0xF4u) { need = 3; hi = 0x8Fu; }
  else return 0;
  if (need >= avail) return 0;
  const uint32_t b1 = s[1];
  if (b1 < lo || b1 > hi) return 0;
  uint32_t v = (b0 & (0x7Fu >> (need + 1))) << 6 | (b1 & 0x3Fu);
  for (int k = 2; k <= need; ++k) {
    const uint32_t bk = s[k];
    if ((bk & 0xC0u) != 0x80u) return 0;
    v = (v << 6) | (bk & 0x3Fu);
  }
  *cp = v;
  return need + 1;
}
#endif

// host-side launchers (defined in the kernel translation units)
void launch_boundaries(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s);
void launch_bpe_engine(const Call& c, const Workspace& w, const DevVocab& v, int n_sms, cudaStream_t s);
void launch_emit(const Call& c, const Workspace& w, const DevVocab& v, cudaStream_t s);
void launch_status_only(const Call& c, const Workspace& w, cudaStream_t s);

__host__ __device__ inline long long n_chunks(long long n) { return (n + CHUNK - 1) / CHUNK; }
__host__ __device__ inline long long n_bchunks(long long n) { return (n + BCHUNK - 1) / BCHUNK; }

}  // namespace tokgb
