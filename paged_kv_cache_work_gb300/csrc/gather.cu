// pa_gather_kv: the paged cache's K and V rows of a batch, copied into two contiguous
// buffers (the copy the HSTU paged attention makes into its workspace before attending,
// "HSTU Paged Attention" K/V double-buffering issue, background and optimisation plan).
//
// A page of a [num_blocks, block_size, Hkv, D] cache is one contiguous run of
// block_size * Hkv * D elements, and so is the stretch of output rows it maps to, so the
// gather is a list of contiguous copies: for each sequence b and page p, the page's first
// min(block_size, n_b - p * block_size) rows of K, then of V.  They are cut into chunks of
// at most kChunk bytes and spread evenly over a persistent grid of one CTA per SM.  One
// thread per CTA moves its chunks through a ring of kStages shared-memory stages with bulk
// copies: a chunk is loaded with cp.async.bulk (completing on the stage's mbarrier), stored
// back with cp.async.bulk into the output (a bulk group), and the stage is refilled as soon
// as the store of the chunk before it has finished reading shared memory, so about kStages
// chunks are always in flight in each direction (the ping-pong of the page's plan, as deep as
// shared memory allows).
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kGatherThreads = 32;
constexpr int kChunk = 16384;        // bytes of one bulk copy
constexpr int kStages = 8;           // ring depth: 128 KB in flight per SM each way
constexpr int kGatherMaxBatch = 8192;  // sequences whose offsets fit in shared memory

struct GatherParams {
  const char* k_cache;
  const char* v_cache;
  char* k_out;
  char* v_out;
  const int32_t* bt;
  const int32_t* ctx;
  int32_t* row_offsets;  // nullable [batch + 1]
  int32_t* flags;        // nullable
  long long max_rows;
  int batch, block_size, max_blocks, num_blocks;
  int row_bytes;       // Hkv * D * bytes per element (a multiple of 16)
  int chunks_full;     // chunks of one full page
};

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Every bulk group but the most recent has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Every bulk group has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Walks the chunks [c, c_end) of the batch in order (sequence, page, K then V, chunk) and
// yields the valid ones; pages with an out-of-range block id are flagged and skipped.
struct ChunkCursor {
  const GatherParams* p;
  const int32_t* s_chunk_off;  // [batch + 1] exclusive prefix of chunks per sequence
  const int32_t* s_row_off;    // [batch + 1] exclusive prefix of rows
  int c, c_end;
  int b, page, kv, k;          // position of chunk c
  int n, full, rem, page_chunks;
  int blk;

  __device__ void set_seq() {
    n = s_row_off[b + 1] - s_row_off[b];
    full = n / p->block_size;
    rem = n - full * p->block_size;
  }
  __device__ int chunks_of_page(int pg) const {
    const int rows = pg < full ? p->block_size : rem;
    return (int)(((long long)rows * p->row_bytes + kChunk - 1) / kChunk);
  }
  __device__ void load_block() {  // the block of the current page (checked once per page)
    blk = __ldg(p->bt + (size_t)b * p->max_blocks + page);
    if ((blk < 0 || blk >= p->num_blocks) && p->flags) atomicOr(p->flags, PA_FLAG_BAD_BLOCK_ID);
  }

  // Position on chunk c0 (0 <= c0 < total).
  __device__ void init(const GatherParams* prm, const int32_t* coff, const int32_t* roff, int c0,
                       int c1) {
    p = prm;
    s_chunk_off = coff;
    s_row_off = roff;
    c = c0;
    c_end = c1;
    if (c >= c_end) return;
    int lo = 0, hi = p->batch;  // last sequence whose chunk offset is <= c
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_chunk_off[mid] <= c) lo = mid + 1; else hi = mid;
    }
    b = lo - 1;
    set_seq();
    int li = c - s_chunk_off[b];
    const int per_full = 2 * p->chunks_full;
    page = li / per_full < full ? li / per_full : full;
    li -= page * per_full;
    page_chunks = chunks_of_page(page);
    kv = li / page_chunks;
    k = li - kv * page_chunks;
    load_block();
  }

  __device__ void advance() {
    ++c;
    if (c >= c_end) return;
    if (++k < page_chunks) return;
    k = 0;
    if (++kv < 2) return;
    kv = 0;
    if (++page >= full + (rem > 0 ? 1 : 0)) {
      // the next sequence with tokens (one exists: chunk c lies inside the batch)
      do {
        ++b;
        set_seq();
      } while (full + (rem > 0 ? 1 : 0) == 0);
      page = 0;
    }
    page_chunks = chunks_of_page(page);
    load_block();
  }

  // The next valid chunk: source, destination and size; false when the range is done.
  __device__ bool next(const char*& src, char*& dst, uint32_t& bytes) {
    while (c < c_end) {
      const bool ok = blk >= 0 && blk < p->num_blocks;
      const int rows = page < full ? p->block_size : rem;
      const long long page_bytes = (long long)rows * p->row_bytes;
      const long long off = (long long)k * kChunk;
      bytes = (uint32_t)(page_bytes - off < kChunk ? page_bytes - off : kChunk);
      src = (kv ? p->v_cache : p->k_cache) +
            ((long long)blk * p->block_size) * p->row_bytes + off;
      dst = (kv ? p->v_out : p->k_out) +
            ((long long)s_row_off[b] + (long long)page * p->block_size) * p->row_bytes + off;
      advance();
      if (ok) return true;
    }
    return false;
  }
};

__global__ void __launch_bounds__(kGatherThreads, 1) gather_kernel(const GatherParams p) {
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  char* ring = smem;                                             // kStages x kChunk
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kStages * kChunk);  // [kStages]
  int32_t* s_row_off = reinterpret_cast<int32_t*>(full + kStages);       // [batch + 1]
  int32_t* s_chunk_off = s_row_off + p.batch + 1;                        // [batch + 1]
  const int lane = threadIdx.x;

  // ---- offsets of every sequence's rows and chunks (each CTA computes them all)
  const long long cap = (long long)p.max_blocks * p.block_size;
  int row_carry = 0, chunk_carry = 0, bad = 0;
  for (int base = 0; base < p.batch; base += 32) {
    const int b = base + lane;
    int n = 0, ch = 0;
    if (b < p.batch) {
      n = __ldg(p.ctx + b);
      if (n < 0 || (long long)n > cap) {
        bad = 1;
        n = 0;
      }
      const int full_pages = n / p.block_size, rem = n - full_pages * p.block_size;
      ch = 2 * (full_pages * p.chunks_full +
                (int)(((long long)rem * p.row_bytes + kChunk - 1) / kChunk));
    }
    int rn = n, rc = ch;  // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yn = __shfl_up_sync(kFull, rn, o), yc = __shfl_up_sync(kFull, rc, o);
      if (lane >= o) {
        rn += yn;
        rc += yc;
      }
    }
    if (b < p.batch) {
      s_row_off[b] = row_carry + rn - n;
      s_chunk_off[b] = chunk_carry + rc - ch;
    }
    row_carry += __shfl_sync(kFull, rn, 31);
    chunk_carry += __shfl_sync(kFull, rc, 31);
  }
  bad = __any_sync(kFull, bad);
  const bool overflow = (long long)row_carry > p.max_rows;
  if (lane == 0) {
    s_row_off[p.batch] = row_carry;
    s_chunk_off[p.batch] = chunk_carry;
    if (blockIdx.x == 0 && p.flags && (bad || overflow)) atomicOr(p.flags, PA_FLAG_BAD_LENGTHS);
  }
  __syncwarp();
  if (blockIdx.x == 0 && p.row_offsets)
    for (int b = lane; b <= p.batch; b += 32) p.row_offsets[b] = s_row_off[b];
  if (overflow) return;  // nothing is copied when the rows do not fit the output
  if (lane != 0) return;

  // ---- this CTA's chunks through the ring (one thread)
  const long long total = chunk_carry;
  const int c0 = (int)(total * blockIdx.x / gridDim.x);
  const int c1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  if (c0 >= c1) return;
  for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
  fence_barrier_init();
  ChunkCursor cur;
  cur.init(&p, s_chunk_off, s_row_off, c0, c1);
  char* dst_of[kStages];
  uint32_t bytes_of[kStages];
  uint32_t nload = 0;
  auto load_next = [&](int s) -> bool {
    const char* src;
    char* dst;
    uint32_t bytes;
    if (!cur.next(src, dst, bytes)) return false;
    dst_of[s] = dst;
    bytes_of[s] = bytes;
    mbar_arrive_expect_tx(&full[s], bytes);
    bulk_load(ring + s * kChunk, src, bytes, &full[s]);
    ++nload;
    return true;
  };
  for (int s = 0; s < kStages; ++s)
    if (!load_next(s)) break;
  volatile int abort_flag = 0;
  uint32_t j = 0;  // the next chunk to store; chunk j sits in stage j % kStages
  for (; j < nload; ++j) {
    const int s = (int)(j % kStages);
    if (!mbar_wait(&full[s], (j / kStages) & 1, &abort_flag)) {
      if (p.flags) atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
      break;
    }
    bulk_store(dst_of[s], ring + s * kChunk, bytes_of[s]);
    if (j >= 1) {  // the store of chunk j - 1 has read its stage: refill it
      bulk_wait_read_all_but_one();
      load_next((int)((j - 1) % kStages));
    }
  }
  bulk_wait_all();
  // loads that were issued but not stored (only after a timeout) land before exit
  for (uint32_t i = j; i < nload; ++i) mbar_wait_drain(&full[i % kStages], (i / kStages) & 1);
}

}  // namespace

size_t gather_smem_bytes(int batch) {
  return 1024 + (size_t)kStages * kChunk + kStages * 8 + 2 * (size_t)(batch + 1) * 4;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_gather_kv(const pa_config* cfg, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  void* k_out, void* v_out, int64_t max_rows,
                                  int32_t* row_offsets, int32_t* flags, cudaStream_t stream) {
  if (!cfg || !k_cache || !v_cache || !block_tables || !context_lens || !k_out || !v_out)
    return PA_ERR_INVALID_ARG;
  const pa_config& c = *cfg;
  if (c.batch < 1 || c.num_kv_heads < 1 || c.max_blocks_per_seq < 1 || c.num_blocks < 1 ||
      max_rows < 0)
    return PA_ERR_INVALID_ARG;
  if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (c.block_size < 16 || c.block_size > 1024 || (c.block_size & (c.block_size - 1)))
    return PA_ERR_UNSUPPORTED;
  if (c.kv_dtype != PA_BF16 && c.kv_dtype != PA_FP16 && c.kv_dtype != PA_FP8_E4M3)
    return PA_ERR_UNSUPPORTED;
  if (c.batch > kGatherMaxBatch) return PA_ERR_UNSUPPORTED;
  auto aligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!aligned(k_cache) || !aligned(v_cache) || !aligned(k_out) || !aligned(v_out))
    return PA_ERR_INVALID_ARG;
  const int bpe = c.kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  const long long row_bytes = (long long)c.num_kv_heads * c.head_dim * bpe;
  if (row_bytes > (1 << 20)) return PA_ERR_UNSUPPORTED;
  const long long page_bytes = row_bytes * c.block_size;
  // offsets are int32 rows and chunk counts
  const long long max_chunks =
      2LL * c.batch * c.max_blocks_per_seq * ((page_bytes + kChunk - 1) / kChunk);
  if ((long long)c.batch * c.max_blocks_per_seq * c.block_size > INT32_MAX ||
      max_chunks > INT32_MAX)
    return PA_ERR_UNSUPPORTED;

  GatherParams p;
  p.k_cache = static_cast<const char*>(k_cache);
  p.v_cache = static_cast<const char*>(v_cache);
  p.k_out = static_cast<char*>(k_out);
  p.v_out = static_cast<char*>(v_out);
  p.bt = block_tables;
  p.ctx = context_lens;
  p.row_offsets = row_offsets;
  p.flags = flags;
  p.max_rows = max_rows;
  p.batch = c.batch;
  p.block_size = c.block_size;
  p.max_blocks = c.max_blocks_per_seq;
  p.num_blocks = c.num_blocks;
  p.row_bytes = (int)row_bytes;
  p.chunks_full = (int)((page_bytes + kChunk - 1) / kChunk);

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ERR_CUDA;
  const size_t smem = gather_smem_bytes(c.batch);
  static std::atomic<uint64_t> attr_done{0};  // devices whose limit is raised
  if (set_smem_attr_once(attr_done, reinterpret_cast<const void*>(gather_kernel),
                         (int)gather_smem_bytes(kGatherMaxBatch)) != cudaSuccess)
    return PA_ERR_CUDA;
  gather_kernel<<<sms, kGatherThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
