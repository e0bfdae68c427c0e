// Merged-weight fast path: W' = W + B A for one adapter, every expert, both
// projections (the hybrid-attention decoder page merges its LoRA into the
// base weights once, with merge_and_unload, so serving pays no LoRA cost).
// Stored layouts: W [E][rows][cols], B [E][rows][r], A [E][r][cols]; W' like W.
//
// HBM-bound: every W element is read once and its W' written once (4 bytes
// per element), and each element needs an r-term dot product -- 2r FLOP per
// 4 bytes, which at r >= 32 is more than CUDA-core FMA keeps up with at HBM
// rate.  So the rank-r product runs on the tensor cores:
//
//  * a tile is 128 rows x 128 columns of one expert; its product
//    D = B_tile (128 x r) . A_tile^T (128 cols x r) is r / 16
//    tcgen05.mma.cta_group::1 (M = 128, N = 128, K = 16) into TMEM (fp32);
//  * a work item is one expert's column block over up to 32 row tiles
//    (the block's row tiles cut into nearly equal ranges): the A_tile^T operand (A is stored r x cols, so the columns are
//    not K-contiguous) is transposed once per item by a dedicated warp into
//    the swizzled K-major layout TMA would give it, one item ahead;
//  * W tiles (two 128 x 64 boxes, 128-byte swizzle) and B tiles come by TMA
//    into a two-slot ring; the epilogue warps add the accumulator row by row
//    to the W tile in shared memory, round once to bf16 in place and write
//    the tile back with a TMA store, so every HBM byte moves in bulk.
//
// Persistent: one CTA per SM, items in a fixed order (expert slow, then the
// row range, column block fast, so the CTAs at work at one time share the
// expert's B and A rows through L2).  No item waits on another CTA.  Every
// wait is bounded; a wait that runs out winds the CTA down (no error word:
// the call has no workspace; the output is then undefined).
#include "common.cuh"
#include "merge.cuh"

#include <algorithm>

namespace moelora {
namespace {

constexpr int kMergeThreads = 352;   // warp 0 TMA, 1 MMA, 2-9 epilogue, 10 A transpose
constexpr int kTile = 128;           // rows and columns of a tile
constexpr int kMaxTilesPerItem = 32; // row tiles of one work item, at most
constexpr int kWBytes = kTile * kTile * 2;       // one W tile (two 64-column boxes)
constexpr int kMaxSlots = 6;                     // ring slots of W and B tiles
// shared memory: barriers (first KB) | W[ns] | B operand (LoRA B rows)[ns] |
// A^T operand[2]; an operand tile is 128 x r bf16.  The ring is as deep as
// the rank leaves room for: 6 slots at r = 16, 5 at 32, 4 at 64, 2 at 128.
constexpr int kBarBytes = 1024;
constexpr int kSmemBudget = 232448 - 1024;        // opt-in maximum less the alignment slack
constexpr int kNumBars = 3 * kMaxSlots + 8;

__host__ __device__ constexpr int merge_slots(int r) {
  return (kSmemBudget - kBarBytes - 2 * kTile * r * 2) / (kWBytes + kTile * r * 2) < kMaxSlots
             ? (kSmemBudget - kBarBytes - 2 * kTile * r * 2) / (kWBytes + kTile * r * 2)
             : kMaxSlots;
}
__host__ __device__ constexpr int merge_smem(int r) {
  return 1024 + kBarBytes + merge_slots(r) * (kWBytes + kTile * r * 2) + 2 * kTile * r * 2;
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// all but the most recent bulk group have read their shared memory
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// 32 lanes x 32 bit, 32 consecutive columns per thread, without waiting:
// several loads can be in flight before one tmem_ld_wait
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// OR of `pred` over the `nthreads` threads of named barrier `id` (the four
// epilogue warps agree on whether to go on).
__device__ __forceinline__ bool bar_any(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

struct MergeItem {
  int e, rt0, nrt, cb;
};

// Item `it`: column block fastest, then the row range (the n_rt row tiles
// of a column block cut into n_rc ranges of nearly equal length), expert
// slowest.
__device__ __forceinline__ MergeItem merge_item(int it, int n_rc, int n_cb, int n_rt) {
  MergeItem m;
  m.cb = it % n_cb;
  const int rest = it / n_cb;
  const int rc = rest % n_rc;
  m.e = rest / n_rc;
  m.rt0 = static_cast<int>(static_cast<long long>(n_rt) * rc / n_rc);
  m.nrt = static_cast<int>(static_cast<long long>(n_rt) * (rc + 1) / n_rc) - m.rt0;
  return m;
}

// Byte offset of element (row n, k) of an operand chunk of width lw (bf16)
// in the K-major layout TMA writes with a (lw * 2)-byte swizzle: 16-byte
// units of a row XORed with the row's position in its 8-row (128-byte
// swizzle), 4-row-pair (64-byte) or 2-row-quad (32-byte) pattern.
__device__ __forceinline__ uint32_t swizzled_off(int n, int k, int lw) {
  const uint32_t off = static_cast<uint32_t>(n * lw * 2 + k * 2);
  const uint32_t mask = lw == 64 ? 7u : (lw == 32 ? 3u : 1u);
  return off ^ (((off >> 7) & mask) << 4);
}

__global__ void __launch_bounds__(kMergeThreads, 1)
    merge_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_wm,
                    const __grid_constant__ CUtensorMap map_b, const __nv_bfloat16* __restrict__ A,
                    int rows, int cols, int r, int lw, int swz, int E) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int ns = merge_slots(r);
  const int op_bytes = kTile * r * 2;              // one operand tile (128 x r)
  uint8_t* w_base = smem + kBarBytes;              // W[ns]
  uint8_t* b_base = w_base + ns * kWBytes;         // B operand[ns]
  uint8_t* a_base = b_base + ns * op_bytes;        // A^T operand[2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* full = bars;                      // [ns] W and B tiles landed
  uint64_t* b_free = bars + kMaxSlots;        // [ns] the MMAs read the B tile
  uint64_t* w_free = bars + 2 * kMaxSlots;    // [ns] the epilogue stored the W tile
  uint64_t* accf = bars + 3 * kMaxSlots;      // [2] accumulator ready
  uint64_t* acce = accf + 2;                  // [2] accumulator read (8 epilogue warps)
  uint64_t* at_full = accf + 4;               // [2] A^T operand written (transpose warp)
  uint64_t* at_free = accf + 6;               // [2] the item's MMAs are done with it
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_rt = (rows + kTile - 1) / kTile;
  const int n_cb = (cols + kTile - 1) / kTile;
  const int n_rc = (n_rt + kMaxTilesPerItem - 1) / kMaxTilesPerItem;
  const int n_items = E * n_rc * n_cb;
  const int chunks = r / lw;                        // operand chunks of lw columns (K)
  const int chunk_bytes = kTile * lw * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&b_free[i]), 1);
      mbar_init(smem_u32(&w_free[i]), 2);   // the stores of both halves
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 8);
      mbar_init(smem_u32(&at_full[i]), 1);
      mbar_init(smem_u32(&at_free[i]), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_wm);
    tma_prefetch_desc(&map_b);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 2 * kTile);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: W and B tiles
    if (lane == 0) {
      uint32_t t = 0;       // tile count of this CTA
      uint32_t posted = 0;  // tiles whose copies were issued
      bool ok = true;
      int s = 0;            // ring slot of tile t, and the phase of its use
      uint32_t sph = 0;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const MergeItem m = merge_item(it, n_rc, n_cb, n_rt);
        for (int i = 0; i < m.nrt && ok; ++i, ++t) {
          if (!(ok = mbar_wait(smem_u32(&b_free[s]), sph ^ 1, abort_flag))) break;
          if (!(ok = mbar_wait(smem_u32(&w_free[s]), sph ^ 1, abort_flag))) break;
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, kWBytes + chunks * chunk_bytes);
          const int row0 = (m.rt0 + i) * kTile;
          const uint32_t wdst = smem_u32(w_base + s * kWBytes);
          tma_load_3d(wdst, &map_w, fb, m.cb * kTile, row0, m.e);
          tma_load_3d(wdst + kWBytes / 2, &map_w, fb, m.cb * kTile + 64, row0, m.e);
          const uint32_t bdst = smem_u32(b_base + s * op_bytes);
          for (int c = 0; c < chunks; ++c)
            tma_load_3d(bdst + c * chunk_bytes, &map_b, fb, c * lw, row0, m.e);
          ++posted;
          if (++s == ns) {
            s = 0;
            sph ^= 1;
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // the copies issued land before the CTA exits (each tile's bytes were
      // announced whole, so its phase completes once they have)
      for (uint32_t u = posted > static_cast<uint32_t>(ns) ? posted - ns : 0; u < posted; ++u) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&full[u % ns]), (u / ns) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t t = 0, item_no = 0;
      bool ok = true, issued = false;
      const uint32_t idesc = make_idesc_bf16(kTile, kTile);
      const uint32_t sbo = static_cast<uint32_t>(8 * lw * 2);
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++item_no) {
        const MergeItem m = merge_item(it, n_rc, n_cb, n_rt);
        const int ab = item_no & 1;
        if (!(ok = mbar_wait(smem_u32(&at_full[ab]), (item_no >> 1) & 1, abort_flag))) break;
        for (int i = 0; i < m.nrt && ok; ++i, ++t) {
          const int s = static_cast<int>(t % ns);     // ring slot
          const int ac = t & 1;                       // accumulator
          if (!(ok = mbar_wait(smem_u32(&full[s]), (t / ns) & 1, abort_flag))) break;
          if (!(ok = mbar_wait(smem_u32(&acce[ac]), ((t >> 1) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t bop = smem_u32(b_base + s * op_bytes);
          const uint32_t aop = smem_u32(a_base + ab * op_bytes);
          uint32_t acc = 0;
          for (int c = 0; c < chunks; ++c) {
            const uint64_t ad = make_smem_desc(bop + c * chunk_bytes, sbo, static_cast<uint32_t>(swz));
            const uint64_t bd = make_smem_desc(aop + c * chunk_bytes, sbo, static_cast<uint32_t>(swz));
            for (int kk = 0; kk < lw / 16; ++kk) {
              mma_bf16(tmem_base + ac * kTile, ad + static_cast<uint64_t>(kk * 2),
                       bd + static_cast<uint64_t>(kk * 2), idesc, acc);
              acc = 1;
            }
          }
          issued = true;
          mma_commit(smem_u32(&b_free[s]));
          mma_commit(smem_u32(&accf[ac]));
          if (i == m.nrt - 1) mma_commit(smem_u32(&at_free[ab]));
        }
      }
      if (!ok) *abort_flag = 1;
      if (issued) {
        // every MMA has completed before TMEM is released
        const uint64_t t0 = globaltimer_ns();
        const uint32_t last = t - 1;
        while (!mbar_try_wait(smem_u32(&accf[last & 1]), (last >> 1) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------ A^T operand, one item ahead
    // lane l takes columns l, l + 32, l + 64, l + 96 of the block; for 8
    // consecutive ranks at a time it gathers one 16-byte K unit per column
    // (loads coalesced across lanes along the row of A) and stores it at its
    // swizzled place
    uint32_t item_no = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x, ++item_no) {
      const MergeItem m = merge_item(it, n_rc, n_cb, n_rt);
      const int ab = item_no & 1;
      if (!(ok = mbar_wait(smem_u32(&at_free[ab]), ((item_no >> 1) & 1) ^ 1, abort_flag))) break;
      uint8_t* dst = a_base + ab * op_bytes;
      const __nv_bfloat16* Ae = A + static_cast<size_t>(m.e) * r * cols;
      for (int q0 = 0; q0 < r; q0 += 8) {
        // ranks q0 .. q0 + 7 of the lane's four columns: 32 loads in flight
        uint16_t h[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = m.cb * kTile + lane + 32 * j;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            h[j][u] = col < cols ? __bfloat16_as_ushort(Ae[static_cast<size_t>(q0 + u) * cols + col]) : 0;
        }
        const int c = q0 / lw;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            v[u] = static_cast<uint32_t>(h[j][2 * u]) | (static_cast<uint32_t>(h[j][2 * u + 1]) << 16);
          *reinterpret_cast<uint4*>(dst + c * chunk_bytes + swizzled_off(lane + 32 * j, q0 - c * lw, lw)) =
              make_uint4(v[0], v[1], v[2], v[3]);
        }
      }
      fence_proxy_async_smem();   // generic-proxy writes, read by the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&at_full[ab]));
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else {
    // ------------------------------------------------ epilogue: W' = W + D, stored by TMA
    // eight warps: warp w takes TMEM lanes 32 (w % 4) .. + 31 (the tile rows
    // its lane quarter may read) and one 64-column half of the tile, which
    // is one TMA box; the four warps of a half store their box together
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;       // row of the tile
    const bool storer = lane == 0 && (warp & 3) == 2;   // warps 2 and 6
    uint32_t t = 0;
    bool ok = true;
    int pending_slot = -1;                     // the slot of this storer's last store
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const MergeItem m = merge_item(it, n_rc, n_cb, n_rt);
      for (int i = 0; i < m.nrt; ++i, ++t) {
        const int s = static_cast<int>(t % ns);
        const int ac = t & 1;
        // the accumulator, and the W tile (complete already: the MMAs were
        // issued after it landed; waited for so that its bytes are visible)
        bool got = mbar_wait(smem_u32(&accf[ac]), (t >> 1) & 1, abort_flag);
        got = got && mbar_wait(smem_u32(&full[s]), (t / ns) & 1, abort_flag);
        if (bar_any(1, 256, !got || *abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* box = w_base + s * kWBytes + half * (kWBytes / 2) + row * 128;
        const uint32_t taddr = tmem_base + ac * kTile + (static_cast<uint32_t>(quarter * 32) << 16) + half * 64;
        float v[64];
        tmem_ld32_nowait(taddr, v);
        tmem_ld32_nowait(taddr + 32, v + 32);
        tmem_ld_wait();
        // the accumulator is read: the MMAs of tile t + 2 may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&acce[ac]));
        // W row `row`, the half's 64 columns: eight 16-byte units at their
        // 128-byte-swizzle places
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4* p = reinterpret_cast<uint4*>(box + ((u ^ (row & 7)) * 16));
          uint4 w = *p;
          uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float a = __uint_as_float(wv[h] << 16) + v[u * 8 + 2 * h];
            const float b = __uint_as_float(wv[h] & 0xffff0000u) + v[u * 8 + 2 * h + 1];
            wv[h] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
          }
          *p = w;
        }
        // the half goes out by TMA; a slot is released once the stores of
        // both halves have read it (checked one tile later, so that the
        // epilogue does not wait for the read)
        fence_proxy_async_smem();
        named_bar_sync(2 + half, 128);
        if (storer) {
          const int x = m.cb * kTile + half * 64;
          if (x < cols)   // (a box wholly past the last column stores nothing)
            tma_store_2d(&map_wm, smem_u32(w_base + s * kWBytes + half * (kWBytes / 2)), x,
                         (m.rt0 + i) * kTile, m.e);
          bulk_commit();
          if (pending_slot >= 0) {
            bulk_wait_read1();
            mbar_arrive(smem_u32(&w_free[pending_slot]));
          }
          pending_slot = s;
        }
      }
    }
    if (!ok) *abort_flag = 1;
    if (storer) {
      bulk_wait0();   // every store has completed
      if (pending_slot >= 0) mbar_arrive(smem_u32(&w_free[pending_slot]));
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kTile);
  }
}

}  // namespace


cudaError_t launch_merge(const CUtensorMap& map_w, const CUtensorMap& map_wm, const CUtensorMap& map_b,
                         const __nv_bfloat16* A, int E, int rows, int cols, int r, int num_sms,
                         cudaStream_t stream) {
  static int configured = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured != dev) {
    cudaError_t e = cudaFuncSetAttribute(merge_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget + 1024);   // covers every rank
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const int lw = r % 64 == 0 ? 64 : (r % 32 == 0 ? 32 : 16);
  const int swz = lw == 64 ? 2 : (lw == 32 ? 4 : 6);   // descriptor layout code of the chunk swizzle
  const int n_rt = (rows + kTile - 1) / kTile;
  const long long n_items = static_cast<long long>(E) *
                            ((n_rt + kMaxTilesPerItem - 1) / kMaxTilesPerItem) * ((cols + kTile - 1) / kTile);
  const int grid = static_cast<int>(std::min<long long>(n_items, num_sms));
  merge_tc_kernel<<<grid, kMergeThreads, merge_smem(r), stream>>>(map_w, map_wm, map_b, A, rows, cols,
                                                                  r, lw, swz, E);
  return cudaGetLastError();
}

}  // namespace moelora
