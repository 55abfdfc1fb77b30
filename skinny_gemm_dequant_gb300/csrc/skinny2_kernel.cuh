// The persistent skinny GEMM kernel (layout, helpers and activation jobs: skinny2.cuh).
//
// One kernel serves three kinds of launch:
//  * S2_DENSE: y = dequant(W) x for INT8 / FP8-block / MXFP4 weights (M <= 16 tokens);
//  * S2_MOE_GU: MoE stage 1 (routing included), for every distinct routed expert e the gate and up rows of W13[e]
//    against all M tokens' activations (the MMA's 8 or 16 token columns cost the same however
//    many are routed); the epilogue keeps the (token, e) pairs the router chose and stores their
//    raw sums gu[pair] in fp32;
//  * S2_MOE_DN: MoE stage 2, for every distinct expert the rows of W2[e] against the gathered
//    rows h = bf16(silu(g) * u) of its pairs (prepared by this kernel's activation jobs from
//    gu); the epilogue stores o[pair] in fp32 for the weighted combine.
// For the MoE kinds a unit is (expert slot, 128-row block, 256 weight bytes of K); the slots are
// the router's distinct experts, so the unit count is read on the device after the
// grid-dependency wait and split evenly over the CTAs there.
#pragma once
#include "skinny2.cuh"

#ifndef QL_LOCAL_MULTI
#define QL_LOCAL_MULTI 1
#endif

namespace ql {

// tmW: 4D view {128 bytes, N rows, full 128-byte chunks, experts} (strides ldw, 128, expert
//      stride), box {128, 128, 2, 1}
// tmW2: 2D view {wbytes, N}, box {128, 128}: dense units holding a partial chunk
// tmX: 4D view of the activation image {64 f16, img_rows, copies, kpad/64}, box {64, Mp, 1, NXB}
//      (rows past img_rows read as zeros)
template <int FMT, int MT, int KIND>
__global__ void __launch_bounds__(S2_THREADS, s2_ctas_per_sm(FMT, MT))
    skinny2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ Skinny2Args a) {
  using Tr = S2Traits<FMT>;
  constexpr int Mp = 8 * MT;
  constexpr uint32_t W_CHUNK = S2_ROWS * 128;  // one 128-byte chunk of all 128 rows (16 KB)
  constexpr uint32_t W_BYTES = W_CHUNK * S2_CHUNKS;
  constexpr uint32_t X_BOX = Mp * 128;         // one 64-element slab of all token rows
  constexpr uint32_t X_BYTES = Tr::NXB * X_BOX;
  constexpr uint32_t STAGE = s2_stage_bytes<FMT, MT>();
  constexpr bool kInt = (FMT == FMT_INT8);
  constexpr bool kMoE = (KIND == S2_MOE_GU || KIND == S2_MOE_DN);
  // local activations (dense layers with few tokens): stages carry weights only and every CTA
  // builds the activation image of its own units behind the barriers (s2_local_image)
  constexpr bool kLocal = (KIND == S2_DENSE_LOCAL);
  constexpr bool kBF16 = (FMT == FMT_BF16);  // activations loaded as they are: no image, no jobs
  constexpr bool kF8C = (FMT == FMT_F8E4C || FMT == FMT_F8E5C);  // FP8 codes, one scale per channel
  constexpr bool kRowScale = kInt || kF8C;                         // fp32 w_scale applied once at the end
  // INT8 dense layers of up to 8 tokens may settle their outputs through cells (exact integer
  // sums, so neither the split nor the order of arrival can change a result); the host asks for
  // it by passing the cells (a.cells)
  constexpr bool kCellCode = kInt && !kMoE && MT == 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  constexpr bool loc = kLocal;
  constexpr uint32_t XB = loc ? 0u : X_BYTES;                 // activation bytes of a stage
  constexpr uint32_t STB = loc ? W_BYTES + Tr::SCB : STAGE;   // stage stride (a multiple of 1 KB)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * STB);
  uint64_t* empty = full + S;
  uint8_t* limg = reinterpret_cast<uint8_t*>(empty + S);  // local activation image (a.local_bytes)
  uint8_t* fp8sc = limg + a.local_bytes;  // FP8 scale rows of this CTA's row blocks
  __shared__ int s_abort;
  __shared__ int s_urb[8], s_ukt[8];  // kDyn: row block and K unit of the stage in each slot (-1: end)
  __shared__ float s_tokf[Mp];         // local activations: the tokens' factors

  // the next kernel in the stream may launch now: it waits for this grid before it touches
  // memory, and meanwhile can take each SM this grid leaves and start streaming its weights
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  if constexpr (!kBF16 && KIND != S2_MOE_DN) {
    // the token rows this CTA's activation jobs will read, into L2 now, while the previous
    // kernel may still run: the loads that use them come after the grid-dependency wait, and
    // a write by the previous kernel lands in L2 all the same (a prefetch changes no value)
    // (local activations: every CTA reads every row)
    if (threadIdx.x == 0)
      for (int j = kLocal ? 0 : c; j < (kLocal ? a.M : a.M * s2_slices(a.M, G, kMoE ? 8 : 32)); j += kLocal ? 1 : G)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a.x + (int64_t)(j % a.M) * a.ldx),
                     "r"((uint32_t)a.K * 2)
                     : "memory");
  }
  // the activation image: the consumer warps of CTAs c, c + G, ... each write one (row, slice)
  // job and count them in with one release (the rows are read by TMA, the async proxy, in other
  // CTAs: proxy fence first; the release is cumulative over the CTA's writes, ordered before it
  // by the barrier)
  __shared__ float s_red[3 * S2_CONSUMERS];  // a job's 8 warp maxima; local multi-token images: 3 per token
  auto run_jobs = [&](int njob_rows, int nsl) {
    unsigned mine = 0;
    for (int j = c; j < njob_rows * nsl; j += G, ++mine) {
      if constexpr (KIND == S2_MOE_DN)
        s2_prepare_h(a, j % njob_rows, j / njob_rows, nsl, threadIdx.x, s_red);
      else
        s2_prepare<FMT>(a, j % njob_rows, j / njob_rows, nsl, threadIdx.x, s_red);
    }
    if (mine) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      consumer_sync();
      if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.ready), "r"(mine) : "memory");
    }
  };
  // MoE: the units follow the distinct routed experts.  gate_up routes here (every CTA alike,
  // into shared memory behind the ring); down reads what gate_up's CTA 0 wrote.  gate_up's
  // activation image needs no routing: its jobs run first, before this grid's weight stream
  // (which starts after routing) competes with their loads and stores.
  int nu = 1;
  const int32_t* r_uniq = a.uniq;  // expert of each slot
  const int32_t* r_ids = a.ids;    // expert of each pair
  if constexpr (kMoE) {
    pdl_wait();
    if constexpr (KIND == S2_MOE_GU) {
      if (warp < S2_CONSUMERS) run_jobs(a.M, s2_slices(a.M, G, 8));
      const int P = a.M * a.topk;
      int* s_ids = reinterpret_cast<int*>(fp8sc);  // no FP8 scale rows for MXFP4
      int* s_cnt = s_ids + P;
      int* s_uniq = s_cnt + a.E + 1;
      int* s_slot = s_uniq + a.E;
      int* s_nu = s_slot + a.E;
      s2_route(a, s_ids, s_cnt, s_uniq, s_slot, s_nu);
      nu = *s_nu;
      r_uniq = s_uniq;
      r_ids = s_ids;
    } else {
      nu = min(*a.nuniq, a.E);
    }
  }
  const int64_t T = kMoE ? (int64_t)nu * a.nb * a.nk : a.total;
  const bool kDyn = kCellCode && a.cells != nullptr;
  const int64_t s0 = (int64_t)c * T / G, s1 = (int64_t)(c + 1) * T / G;
  const int nk = a.nk;
  const uint32_t lim = a.wait_limit;
  volatile int* abort = &s_abort;
  auto fail = [&]() {
    atomicOr(a.status, (uint32_t)QL_DEV_TIMEOUT);
    *abort = 1;
  };
  // jobs that build the activation image, and how many of them the producers wait for
  const int njob_rows = KIND == S2_MOE_DN ? a.offsets[a.E] : (kBF16 ? 0 : a.M);
  const int nsl = s2_slices(max(njob_rows, 1), G, kMoE ? 8 : 32);
  const unsigned need = (unsigned)(njob_rows * nsl);

  const int rb_first = (int)(s0 / nk);  // global row block (expert slot * nb + block)
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], FMT == FMT_MXFP4 ? 1 + 32 : 1);
      tc::mbar_init(&empty[i], S2_CONSUMERS);
    }
    tc::fence_mbar_init();
    s_abort = 0;
    if constexpr (kLocal)
      for (int i = 0; i < 8; ++i) s_red[i] = 0.f;  // multi-token local images: per-token amax maxima
    tc::tma_prefetch_desc(&tmW);
    tc::tma_prefetch_desc(&tmX);
  }
  if constexpr (FMT == FMT_FP8) {  // dense only: the block-scale rows of this CTA's row blocks
    const int nbr = S2_ROWS / a.block_n + 2;  // n-blocks a 128-row block can touch
    const int rb_last = (int)((s1 - 1) / nk);
    const int nrow_blocks = rb_last - rb_first + 1;
    const int nb0 = (rb_first * S2_ROWS) / a.block_n;
    const int nb_count = min(nrow_blocks * nbr, (int)((a.N + a.block_n - 1) / a.block_n) - nb0);
    for (int i = threadIdx.x; i < nb_count * a.lds; i += blockDim.x) fp8sc[i] = a.wsb[(int64_t)nb0 * a.lds + i];
  }
  __syncthreads();

  if (warp == S2_CONSUMERS) {
    // ------------------------------------------------------------ producer warp
    const int n_units = (int)(s1 - s0);
    const int pre = min(S, n_units);
    const int xcp = c % a.xcopies;  // this CTA's copy of the activation image
    const bool whole_chunks = (a.wbytes & 127) == 0;
    const int ksc = a.K / 32;  // MXFP4 scale bytes of a row that belong to K
    // the activation hand-off: wait (bounded) until the image is complete, count in (the last
    // producer returns both counters to zero for the next call) and report whether it timed out
    auto handoff_wait = [&]() {
      pdl_wait();  // the counters belong to the previous call until its grid is done
      for (uint32_t n = 0;; ++n) {
        unsigned v;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a.ready) : "memory");
        if (v >= need) break;
        if (n >= lim) {
          fail();
          break;
        }
        __nanosleep(32);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> TMA reads
    };
    // counted in after the activation loads went out (its round trip is off the critical path)
    auto handoff_count = [&]() {
      if (atomicAdd(a.done, 1u) == (unsigned)G - 1) {
        *a.ready = 0;
        *a.done = 0;
      }
    };
    auto handoff = [&]() {
      handoff_wait();
      handoff_count();
    };
    if (n_units == 0) {
      if (lane == 0 && !kBF16 && !loc) handoff();
      if (lane == 0 && kCellCode && kDyn) {  // the consumers wait for an end marker
        s_urb[0] = -1;
        tc::mbar_arrive(&full[0]);
      }
      return;
    }
    // activation tiles of unit kt: the image (4D) or, for BF16, the caller's x itself (2D boxes
    // of 64 columns, rows past M and columns past K read as zeros)
    auto load_x = [&](uint32_t dst, int ktx, int xrow_, uint64_t* bar) {
      if constexpr (kBF16) {
#pragma unroll
        for (int j = 0; j < Tr::NXB; ++j)
          tc::tma_load_2d(smem + (dst - tc::smem_u32(smem)) + j * X_BOX, &tmX, (ktx * Tr::NXB + j) * 64, 0, bar);
      } else {
        tma_load_4d(dst, &tmX, 0, xrow_, xcp, ktx * Tr::NXB, bar);
      }
    };
    if (kCellCode && kDyn) {
      // INT8 through the cells: this CTA's range, its first stages before the hand-off, each
      // stage tagged with its row block and K unit for the consumers.  Lane 0 does all of it.
      if (lane != 0) return;
      const int pre_s = min(S, n_units);
      const uint64_t wpol = tc::l2_evict_first();
      bool ok = true;
      int issued = 0, slot = 0;
      uint32_t phase = 0;
      int urb = rb_first, ukt = (int)(s0 - (int64_t)rb_first * nk);
      for (int i = 0; i <= n_units; ++i) {
        if (i >= S && !tc::mbar_wait(&empty[slot], phase ^ 1u, lim, abort)) {
          fail();
          ok = false;
          break;
        }
        if (i == n_units) {  // no more units: tell the consumers
          s_urb[slot] = -1;
          tc::mbar_arrive(&full[slot]);
          break;
        }
        s_urb[slot] = urb;
        s_ukt[slot] = ukt;
        const uint32_t st = tc::smem_u32(smem + (size_t)slot * STB);
        tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + XB);
        if (whole_chunks || (ukt + 1) * S2_WB <= a.wbytes) {
          tma_load_4d_hint(st, &tmW, 0, urb * S2_ROWS, ukt * S2_CHUNKS, 0, &full[slot], wpol);
        } else {
          tc::tma_load_2d(smem + (size_t)slot * STB, &tmW2, ukt * S2_WB, urb * S2_ROWS, &full[slot]);
          tc::tma_load_2d(smem + (size_t)slot * STB + W_CHUNK, &tmW2, ukt * S2_WB + 128, urb * S2_ROWS, &full[slot]);
        }
        if (loc) {
          // activations are the consumers' own: nothing to load, no hand-off
        } else if (i >= pre_s) {
          load_x(st + W_BYTES, ukt, 0, &full[slot]);
        } else if (i == pre_s - 1) {
          // the stages so far went out without their activations: wait for the image, then
          // load those
          handoff_wait();
          int kj = (int)(s0 - (int64_t)rb_first * nk);
          for (int j = 0; j < pre_s; ++j) {
            load_x(tc::smem_u32(smem + (size_t)j * STB) + W_BYTES, kj, 0, &full[j]);
            if (++kj == nk) kj = 0;
          }
          handoff_count();
        }
        issued = i + 1;
        if (++ukt == nk) {
          ukt = 0;
          ++urb;
        }
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {  // no copy may land after the CTA exits
        for (int i = max(0, issued - S); i < issued; ++i)
          tc::mbar_wait(&full[i % S], (uint32_t)(i / S) & 1, 1u << 22, nullptr);
      }
      return;
    }
    bool ok = true;
    int issued = 0;
    // weights are read once: they leave L2 first, before activations, scales and outputs
    const uint64_t wpol = tc::l2_evict_first();
    // unit counters kept incrementally: no divisions in the loop
    int rb = rb_first, kt = (int)(s0 - (int64_t)rb_first * nk);
    int u = kMoE ? rb / a.nb : 0, rbl = rb - u * a.nb;  // expert slot, block within the expert
    int ex = kMoE ? r_uniq[u] : 0;                      // expert
    int slot = 0;
    uint32_t phase = 0;  // (i / S) & 1
    for (int i = 0; i < n_units; ++i) {
      int got = 1;
      if (lane == 0 && i >= S) got = tc::mbar_wait(&empty[slot], phase ^ 1u, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        ok = false;
        break;
      }
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STB);
      const int xrow = KIND == S2_MOE_DN ? u * a.slot_rows : 0;  // first image row of this unit
      if (lane == 0) {
        // weights: chunks 2kt, 2kt+1 of rows rbl*128.. of expert ex -> smem [chunk][row][128 B]
        if (whole_chunks || (kt + 1) * S2_WB <= a.wbytes) {
          tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + XB);
          tma_load_4d_hint(st, &tmW, 0, rbl * S2_ROWS, kt * S2_CHUNKS, ex, &full[slot], wpol);
        } else {
          // the row ends inside this unit, off a chunk boundary: a chunk at a time from the 2D
          // view, whose bytes past the end (a whole chunk, possibly) are filled with zeros
          tc::mbar_arrive_expect_tx(&full[slot], W_BYTES + XB);
          tc::tma_load_2d(smem + (size_t)slot * STB, &tmW2, kt * S2_WB, rbl * S2_ROWS, &full[slot]);
          tc::tma_load_2d(smem + (size_t)slot * STB + W_CHUNK, &tmW2, kt * S2_WB + 128, rbl * S2_ROWS, &full[slot]);
        }
        if (loc) {
          // activations are the consumers' own: nothing to load, no hand-off
        } else if (i >= pre) {
          load_x(st + W_BYTES, kt, xrow, &full[slot]);
        } else if (i == pre - 1) {
          // the activation image is written by this grid's consumer warps: wait for it, then
          // load the activation tiles of the stages already in flight.  On a timeout the
          // status is flagged and the loads still go out, so no stage waits forever.
          if constexpr (kBF16)
            pdl_wait();  // x may come from the previous kernel
          else
            handoff_wait();
          int ktj = (int)(s0 - (int64_t)rb_first * nk), rbj = rb_first;
          for (int j = 0; j < pre; ++j) {  // pre <= S: stage j is slot j
            const int uj = kMoE ? rbj / a.nb : 0;
            const uint32_t stj = tc::smem_u32(smem + (size_t)j * STB);
            load_x(stj + W_BYTES, ktj, KIND == S2_MOE_DN ? uj * a.slot_rows : 0, &full[j]);
            if (++ktj == nk) {
              ktj = 0;
              ++rbj;
            }
          }
          if constexpr (!kBF16) handoff_count();
        }
      }
      if constexpr (FMT == FMT_MXFP4) {
        // per-32 scale bytes of the unit: 128 rows x (8 bytes per chunk); bytes past K read as 0
        const uint32_t sc = st + W_BYTES + XB;
        const uint8_t* sbase = a.wsb + (int64_t)ex * a.s_estride;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = lane * 4 + (j >> 1), h = j & 1;
          const int n = min(rbl * S2_ROWS + r, a.N - 1);
          const int b0 = kt * 16 + h * 8;
          cp_async8(sc + r * 16 + h * 8, sbase + (int64_t)n * a.lds + (b0 < ksc ? b0 : 0), b0 < ksc ? 8u : 0u);
        }
        cp_async_mbar_arrive(&full[slot]);
      }
      issued = i + 1;
      if (++kt == nk) {
        kt = 0;
        ++rb;
        if (++rbl == a.nb) {
          rbl = 0;
          ++u;
          if (kMoE && u < nu) ex = r_uniq[u];
        }
      }
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      // no copy may land after the CTA exits: wait for every stage still in flight
      for (int i = max(0, issued - S); i < issued; ++i)
        tc::mbar_wait(&full[i % S], (uint32_t)(i / S) & 1, 1u << 22, nullptr);
    }
    if constexpr (FMT == FMT_MXFP4) asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  // -------------------------------------------------------------- consumer warps
  // activations may come from the previous kernel in the stream: wait for it, then write this
  // CTA's jobs of the activation image (gate_up wrote them before routing)
  pdl_wait();
  const int kt0c = (int)(s0 - (int64_t)rb_first * nk);  // K unit of this CTA's first unit
  if constexpr (kLocal) {
#if QL_LOCAL_MULTI
    // one pass over all rows when it takes fewer rounds of eight loads per thread than the
    // token-by-token build takes tokens (measured: 4 tokens x K = 5120 -0.8 us a call, 2 tokens x
    // K = 17408 +0.8 us)
    if (a.M > 1 && (a.K / 8 * a.M + 2047) / 2048 < a.M)
      s2_local_image_multi<FMT>(a, tc::smem_u32(limg), kt0c, (int)min(s1 - s0, (int64_t)nk), threadIdx.x, s_red,
                                s_tokf);
    else
#endif
      s2_local_image<FMT>(a, tc::smem_u32(limg), kt0c, (int)min(s1 - s0, (int64_t)nk), threadIdx.x, s_red, s_tokf);
  }
  else if constexpr (KIND != S2_MOE_GU)
    run_jobs(njob_rows, nsl);
  const int g = lane >> 2, t = lane & 3;
  const int gx = s2_rho(g);  // the activation row this thread's MMA column reads
  const int w = warp;  // 16-row tile of the unit
  // ldmatrix addressing: lane L feeds row 16w + (L & 7) + 8*((L >> 3) & 1) of piece 2p + (L >> 4)
  const int lrow = 16 * w + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int lpc = lane >> 4;
  // activation tiles: the stage's (TMA-loaded) or, with local activations, slot kt - kt0 of the
  // CTA's own image, whose slabs hold only the M real rows (a thread's row is clamped to M - 1:
  // the columns of padding tokens are never stored)
  const uint32_t xsl = kLocal ? (uint32_t)(a.M * 128) : X_BOX;  // bytes between 64-K slabs
  const uint32_t lslot = (uint32_t)(Tr::NXB * a.M * 128);
  const uint32_t limg_s = tc::smem_u32(limg);
  int xr_[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) xr_[m] = kLocal ? min(gx + 8 * m, a.M - 1) : gx + 8 * m;
  auto xtile = [&](uint32_t st, int ktu) -> uint32_t {
    if constexpr (!kLocal) {
      return st + W_BYTES;
    } else {
      int sl = ktu - kt0c;
      if (sl < 0) sl += nk;
      return limg_s + (uint32_t)sl * lslot;
    }
  };
  const float* tokf_p = kLocal ? s_tokf : a.tokf;  // the tokens' factors (x_s or 2^p)

  if (kCellCode && kDyn) {
    // INT8 units as the producer hands them over (slot -> row block, K unit).  A run of
    // consecutive units of one row block is summed in registers (exact int32); when the run
    // ends its sums go out as one atomic add per output cell (s2_cell_add), whose result is
    // inspected at the end of the next run, so the round trip overlaps that run's work: the add
    // that completed a cell's unit count settles the output, y = bf16((acc * x_s) * w_s) (+ bias
    // after the cast).  Every cell starts the call at zero: left so by the previous call (the
    // cell is reset once it has settled) or zeroed by the activation jobs before the hand-off,
    // which no stage reaches a consumer before.
    int32_t acci[MT][4];
    unsigned long long pend[MT][4];  // cell values after this warp's last adds
    int pend_rb = -1;                // their row block (-1: none outstanding)
    int cur_rb = -1, last_kt = -2, run = 0;
    const int row_g = 16 * w + g;
    auto zero = [&]() {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) acci[m][r] = 0;
    };
    auto settle = [&]() {  // the outputs whose unit count the last adds completed
      if (pend_rb < 0) return;
      // the epilogue's factors first, so their loads overlap the adds' round trip
      float xs[MT][2], wsr[2], bsr[2];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int col = s2_rho(2 * t + e2) + 8 * m;
          xs[m][e2] = col < a.M ? tokf_p[col] : 0.f;
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = min(pend_rb * S2_ROWS + row_g + 8 * h, a.N - 1);
        wsr[h] = a.w_scale ? a.w_scale[a.w_scale_len > 1 ? row : 0] : 0.f;
        bsr[h] = a.bias ? bf16_bits_to_f32(a.bias[row]) : 0.f;
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = s2_rho(2 * t + (r & 1)) + 8 * m;
          const int row = pend_rb * S2_ROWS + row_g + (r >= 2 ? 8 : 0);
          if (row >= a.N || col >= a.M || s2_cell_units(pend[m][r]) != nk) continue;
          const int32_t v = s2_cell_sum(pend[m][r]);
          if (a.cells_clean) a.cells[(int64_t)col * a.N + row] = 0ull;  // every add has arrived
          if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = v;
          if (!a.y) continue;  // a K shard: the int32 sums are the result
          uint16_t yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)v, xs[m][r & 1]), wsr[r >> 1]));
          if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + bsr[r >> 1]);
          a.y[(int64_t)col * a.ldy + row] = yb;
        }
      pend_rb = -1;
    };
    auto post = [&]() {  // the run's sums to their cells
      settle();
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = s2_rho(2 * t + (r & 1)) + 8 * m;
          const int row = cur_rb * S2_ROWS + row_g + (r >= 2 ? 8 : 0);
          if (row >= a.N || col >= a.M) continue;
          const unsigned long long add = s2_cell_add(run, acci[m][r]);
          pend[m][r] = atomicAdd(a.cells + (int64_t)col * a.N + row, add) + add;
        }
      pend_rb = cur_rb;
      run = 0;
      zero();
    };
    zero();
    int slot = 0;
    uint32_t phase = 0;
    volatile int* vurb = s_urb;
    volatile int* vukt = s_ukt;
    while (true) {
      int got = 0;
      if (lane == 0) got = tc::mbar_wait(&full[slot], phase, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) fail();
        return;  // the outputs of an aborted call are undefined (the status word says so)
      }
      const int urb = vurb[slot];
      if (urb < 0) break;
      const int ukt = vukt[slot];
      if (run > 0 && (urb != cur_rb || ukt != last_kt + 1)) post();
      cur_rb = urb;
      last_kt = ukt;
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STB);
      const uint32_t xt = xtile(st, ukt);
      float ui[2][MT][4];  // two fp32 chains: integers below 2^24, exact
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int m = 0; m < MT; ++m) ui[e][m][0] = ui[e][m][1] = ui[e][m][2] = ui[e][m][3] = 0.f;
#pragma unroll
      for (int ck = 0; ck < S2_CHUNKS; ++ck) {
        const uint32_t wt = st + ck * W_CHUNK;
        uint32_t q[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          ldmatrix_x4(wt + sw128(lrow, (2 * p + lpc) * 16), q[p][0], q[p][1], q[p][2], q[p][3]);
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
          uint32_t a0, a1, a2, a3;
          s8x4_to_f16x2x2(qa, a0, a2);
          s8x4_to_f16x2x2(qb, a1, a3);
          const int kx = 16 * pc + 4 * t;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * xsl + sw128(xr_[m], (kx & 63) * 2));
            mma_f16_16816(ui[pc & 1][m], a0, a1, a2, a3, xv.x, xv.y);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) acci[m][r] += __float2int_rn(ui[0][m][r] + ui[1][m][r]);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      ++run;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (run > 0) post();
    settle();
    return;
  }

  // one complete row block's results (fp32 sums, or int32 bits for INT8) to their outputs.  The
  // per-token factors (x_s or 2^p) are read here: a stage has arrived by then, and activations
  // were loaded only after the image, factors included, was complete.
  auto emit = [&](int grb, const float (&res)[MT][4]) {
    const int eu = kMoE ? grb / a.nb : 0;  // expert slot
    const int row_w = (grb - eu * a.nb) * S2_ROWS + 16 * w;
    const int ex = kMoE ? r_uniq[eu] : 0;
    int beg = 0, cnt = a.M;  // MoE down: the expert's pairs are dispatch positions beg..beg+cnt-1
    if constexpr (KIND == S2_MOE_DN) {
      beg = a.offsets[ex];
      cnt = min(a.offsets[ex + 1] - beg, a.slot_rows);
    }
    float colf[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int col = s2_rho(2 * t + e2) + 8 * m;  // the token of MMA column 2t + e2
        colf[m][e2] = col < cnt ? (kBF16 ? 1.f : tokf_p[(KIND == S2_MOE_DN ? eu * a.slot_rows : 0) + col]) : 0.f;
      }
    float rowf[2] = {1.f, 1.f}, rowb[2] = {0.f, 0.f};
    if constexpr (!kMoE) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int row = min(row_w + g + 8 * e2, a.N - 1);
        if (kRowScale && a.w_scale) rowf[e2] = a.w_scale[a.w_scale_len > 1 ? row : 0];
        if (a.bias) rowb[e2] = bf16_bits_to_f32(a.bias[row]);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int col = s2_rho(2 * t + (r & 1)) + 8 * m;  // token
        const int row = row_w + g + (r >= 2 ? 8 : 0);
        if (row >= a.N || col >= cnt) continue;
        if constexpr (KIND == S2_MOE_GU) {
          // keep the sums of the pair (token col, expert ex), if the router chose it
          int p = -1;
          for (int k = 0; k < a.topk; ++k)
            if (r_ids[col * a.topk + k] == ex) p = col * a.topk + k;
          if (p >= 0) a.gu[(int64_t)p * a.N + row] = res[m][r] * colf[m][r & 1];
        } else if constexpr (KIND == S2_MOE_DN) {
          a.o[(int64_t)a.pairs[beg + col] * a.N + row] = res[m][r] * colf[m][r & 1];
        } else {
          uint16_t yb;
          if constexpr (kInt) {
            const int32_t v = __float_as_int(res[m][r]);
            if (a.acc_out) a.acc_out[(int64_t)col * a.N + row] = v;
            if (!a.y) continue;  // a K shard: the int32 sums are the result
            yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn((float)v, colf[m][r & 1]), rowf[r >> 1]));
          } else if constexpr (kF8C) {
            yb = f32_to_bf16_rn(__fmul_rn(__fmul_rn(res[m][r], colf[m][r & 1]), rowf[r >> 1]));
          } else {
            if (a.y32) {  // a K shard: the fp32 partial sum, rounded once after the reduction
              a.y32[(int64_t)col * a.ldy32 + row] = res[m][r] * colf[m][r & 1];
              continue;
            }
            yb = f32_to_bf16_rn(res[m][r] * colf[m][r & 1]);
          }
          if (a.bias) yb = f32_to_bf16_rn(bf16_bits_to_f32(yb) + rowb[r >> 1]);
          a.y[(int64_t)col * a.ldy + row] = yb;
        }
      }
  };

  float acc[MT][4];
  int32_t acci[MT][4];
  float own[MT][4];  // partial sums of the block this CTA settles
  int settle_rb = -1;
  bool ok = true;
  int rb = rb_first;
  int kt = (int)(s0 - (int64_t)rb_first * nk);
  int slot = 0;
  uint32_t phase = 0;
  int left = (int)(s1 - s0);  // units still to consume
  while (left > 0) {
    const int kt0 = kt;
    const int seg_units = min(nk - kt, left);  // this row block's units in the range
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        acc[m][r] = 0.f;
        acci[m][r] = 0;
      }
    const uint8_t* sc_row = nullptr;  // FP8 (dense): scale row of this warp's n-block
    if constexpr (FMT == FMT_FP8) {
      const int nb = min(rb * S2_ROWS + 16 * w, a.N - 1) / a.block_n;
      sc_row = fp8sc + (int64_t)(nb - (rb_first * S2_ROWS) / a.block_n) * a.lds;
    }
    for (int u = 0; u < seg_units; ++u, ++kt) {
      int got = 0;
      if (lane == 0 && ok) got = tc::mbar_wait(&full[slot], phase, lim, abort);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        // timed out (or another role did): stop computing but keep walking the units, so
        // every consumer warp still reaches the same named barriers below
        if (lane == 0 && ok) fail();
        ok = false;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        continue;
      }
      const uint32_t st = tc::smem_u32(smem + (size_t)slot * STB);
      const uint32_t xt = xtile(st, kt);
      // INT8 and per-channel FP8: the unit's sums in two fp32 chains.  For INT8 every partial sum
      // is an integer of at most 256 x 127 x 127 < 2^24 in magnitude, so they are exact and
      // convert once per unit
      float ui[2][MT][4];
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int m = 0; m < MT; ++m) ui[e][m][0] = ui[e][m][1] = ui[e][m][2] = ui[e][m][3] = 0.f;
#pragma unroll
      for (int ck = 0; ck < S2_CHUNKS; ++ck) {
        const uint32_t wt = st + ck * W_CHUNK;
        // the chunk's 8 sixteen-byte pieces for this warp's 16 rows (4 ldmatrix.x4):
        // q[p] = (row g, piece 2p), (g+8, 2p), (g, 2p+1), (g+8, 2p+1)
        uint32_t q[4][4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          ldmatrix_x4(wt + sw128(lrow, (2 * p + lpc) * 16), q[p][0], q[p][1], q[p][2], q[p][3]);
        if constexpr (FMT == FMT_BF16) {
          // bf16 weights: q[p] is already the A fragment of the MMA over K 16p..16p+15 of the
          // chunk (64 K = one activation slab); tokens' x at K 16p+2t.. and 16p+8+2t..
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint32_t xs = xt + ck * xsl;
              const uint32_t b0 = lds32(xs + sw128(xr_[m], 32 * p + 4 * t));
              const uint32_t b1 = lds32(xs + sw128(xr_[m], 32 * p + 16 + 4 * t));
              mma_bf16_16816(acc[m], q[p][0], q[p][1], q[p][2], q[p][3], b0, b1);
            }
        } else if constexpr (FMT == FMT_MXFP4) {
          // scale bytes of rows g and g+8 for the chunk's 8 groups
          const uint32_t sbase = st + W_BYTES + XB;
          const uint2 sa8 = lds64(sbase + (16 * w + g) * 16 + ck * 8);
          const uint2 sb8 = lds64(sbase + (16 * w + g + 8) * 16 + ck * 8);
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {  // piece = one 32-element scale group
            const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
            // this thread's 8 weights of the piece are K 8t..8t+7: the activations of those
            // K are 16 contiguous bytes of the token's row
            const int kx = 32 * pc + 8 * t;  // K within the chunk
            uint4 xv[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m)
              xv[m] = lds128(xt + (4 * ck + (kx >> 6)) * xsl + sw128(xr_[m], (kx & 63) * 2));
            float blk[MT][4];
#pragma unroll
            for (int m = 0; m < MT; ++m) blk[m][0] = blk[m][1] = blk[m][2] = blk[m][3] = 0.f;
            uint32_t wa[4], wb[4];  // bytes 0..3 of rows g and g+8 as f16 pairs
            e2m1x8_to_f16x2x4(qa, wa);
            e2m1x8_to_f16x2x4(qb, wb);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int m = 0; m < MT; ++m)
                mma_f16_16816(blk[m], wa[2 * h], wb[2 * h], wa[2 * h + 1], wb[2 * h + 1], h ? xv[m].z : xv[m].x,
                              h ? xv[m].w : xv[m].y);
            // the group's scale bytes of rows g (byte 0) and g+8 (byte 1), decoded together
            uint32_t two;
            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(two) : "r"(pc < 4 ? sa8.x : sa8.y), "r"(pc < 4 ? sb8.x : sb8.y),
                "r"((uint32_t)(((4 + (pc & 3)) << 4) | (pc & 3))));
            const float2 fab = ue8m0x2_to_f32x2(two);
            const float fa = fab.x, fb = fab.y;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              acc[m][0] = fmaf(blk[m][0], fa, acc[m][0]);
              acc[m][1] = fmaf(blk[m][1], fa, acc[m][1]);
              acc[m][2] = fmaf(blk[m][2], fb, acc[m][2]);
              acc[m][3] = fmaf(blk[m][3], fb, acc[m][3]);
            }
          }
        } else if constexpr (kF8C) {
          // FP8 codes to exact f16 and straight into the unit's two fp32 chains: the channel
          // scale is applied once, in the epilogue
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {
            const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
            uint32_t a0, a1, a2, a3;
            if constexpr (FMT == FMT_F8E4C) {
              e4m3x4_to_f16x2x2(qa, a0, a2);
              e4m3x4_to_f16x2x2(qb, a1, a3);
            } else {
              e5m2x4_to_f16x2x2(qa, a0, a2);
              e5m2x4_to_f16x2x2(qb, a1, a3);
            }
            const int kx = 16 * pc + 4 * t;  // K within the chunk of this thread's 4 weights
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * xsl + sw128(xr_[m], (kx & 63) * 2));
              mma_f16_16816(ui[pc & 1][m], a0, a1, a2, a3, xv.x, xv.y);
            }
          }
        } else if constexpr (FMT == FMT_INT8) {
#pragma unroll
          for (int pc = 0; pc < 8; ++pc) {
            const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
            uint32_t a0, a1, a2, a3;
            s8x4_to_f16x2x2(qa, a0, a2);
            s8x4_to_f16x2x2(qb, a1, a3);
            const int kx = 16 * pc + 4 * t;  // K within the chunk of this thread's 4 weights
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * xsl + sw128(xr_[m], (kx & 63) * 2));
              mma_f16_16816(ui[pc & 1][m], a0, a1, a2, a3, xv.x, xv.y);
            }
          }
        } else {
#pragma unroll
          // the chunk's 128 K in two 64-K halves; with blocks of 128 K or more the whole chunk
          // shares one scale and folds once, else each half folds with its own
          const bool whole = a.bk_shift >= 7;
          float blk[2][MT][4];  // two chains so consecutive MMAs are independent
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int m = 0; m < MT; ++m) blk[e][m][0] = blk[e][m][1] = blk[e][m][2] = blk[e][m][3] = 0.f;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int pc = 4 * hb + j;
              const uint32_t qa = q[pc >> 1][2 * (pc & 1)], qb = q[pc >> 1][2 * (pc & 1) + 1];
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16x2x2(qa, a0, a2);
              e4m3x4_to_f16x2x2(qb, a1, a3);
              const int kx = 16 * pc + 4 * t;  // K within the chunk of this thread's 4 weights
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const uint2 xv = lds64(xt + (2 * ck + (kx >> 6)) * xsl + sw128(xr_[m], (kx & 63) * 2));
                mma_f16_16816(blk[j & 1][m], a0, a1, a2, a3, xv.x, xv.y);
              }
            }
            if (hb == 1 || !whole) {
              const int k0 = (kt * S2_CHUNKS + ck) * 128 + (whole ? 0 : 64 * hb);  // first K folded
              // block_k is a power of two; K past the last block (zero weights) has no scale byte
              const float f = k0 < a.K ? ue8m0_to_f32(sc_row[min(k0, a.K - 1) >> a.bk_shift]) : 0.f;
#pragma unroll
              for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                  acc[m][r] = fmaf(blk[0][m][r] + blk[1][m][r], f, acc[m][r]);
                  blk[0][m][r] = blk[1][m][r] = 0.f;
                }
            }
          }
        }
      }
      if constexpr (FMT == FMT_INT8) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) acci[m][r] += __float2int_rn(ui[0][m][r] + ui[1][m][r]);
      } else if constexpr (kF8C) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[m][r] += ui[0][m][r] + ui[1][m][r];
      }
      // every shared-memory fragment of the unit has been read: hand the stage back
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    left -= seg_units;

    // ------------------------------------------------------------ row-block (segment) end
    float res[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) res[m][r] = kInt ? __int_as_float(acci[m][r]) : acc[m][r];
    const int kt_end = kt;
    const int seg_rb = rb;
    rb += 1;  // the next segment (if any) starts a new row block
    kt = 0;
    if (kt0 == 0 && kt_end == nk) {
      emit(seg_rb, res);
      continue;
    }
    const int cf = s2_cta_of((int64_t)seg_rb * nk, T, G);
    if (c == cf) {
      // this CTA settles the block after its last unit (this is its last segment)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) own[m][r] = res[m][r];
      settle_rb = seg_rb;
      continue;
    }
    // another CTA settles it: store the partial sums in this CTA's slot (a CTA posts at most
    // once: for its first segment), then count in with release order
    float* pb = a.part + (int64_t)c * Mp * S2_ROWS;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int col = 2 * t + (r & 1) + 8 * m;
        const int rl = 16 * w + g + (r >= 2 ? 8 : 0);
        pb[col * S2_ROWS + rl] = res[m][r];
      }
    __threadfence();
    consumer_sync();
    if (threadIdx.x == 0) atomicAdd(&a.tickets[seg_rb], 1u);
  }

  // -------------------------------------------------------------- settle the shared block
  if (settle_rb >= 0) {
    const int grb = settle_rb;
    const int cl = s2_cta_of((int64_t)grb * nk + nk - 1, T, G);
    const int count = cl - c + 1;
    // the other CTAs' partial sums: wait (bounded) until all count-1 of them are in
    if (threadIdx.x == 0) {
      uint32_t n = 0;
      while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a.tickets + grb) : "memory");
        if (v >= (unsigned)(count - 1)) break;
        if (++n > lim || *abort) {
          fail();
          break;
        }
        __nanosleep(64);
      }
    }
    consumer_sync();
    // this CTA's sums first, then CTAs c+1..cl in order, four slots' loads in flight at a time
    float sum[MT][4];
    int32_t sumi[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        sum[m][r] = own[m][r];
        sumi[m][r] = __float_as_int(own[m][r]);
      }
    for (int u0 = 1; u0 < count; u0 += 4) {
      float v[MT][4][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = 2 * t + (r & 1) + 8 * m;
          const int rl = 16 * w + g + (r >= 2 ? 8 : 0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            v[m][r][k] = (u0 + k < count) ? __ldcg(a.part + ((int64_t)(c + u0 + k) * Mp + col) * S2_ROWS + rl) : 0.f;
        }
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (u0 + k >= count) break;
            if (kInt)
              sumi[m][r] += __float_as_int(v[m][r][k]);
            else
              sum[m][r] += v[m][r][k];
          }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < 4; ++r) sum[m][r] = kInt ? __int_as_float(sumi[m][r]) : sum[m][r];
    emit(grb, sum);
    if (threadIdx.x == 0) a.tickets[grb] = 0;  // ready for the next call
  }
}

}  // namespace ql
