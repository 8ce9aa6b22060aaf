// schedule.cuh -- which 16-token chunks each decode worker (one warp) handles.
//
// All chunks of the batch are laid end to end: sequence-major, then KV head
// (and query sub-group), then chunk.  The first part of that order is split
// into equal contiguous static ranges, one per worker; the rest is cut into
// small dynamic tiles that workers take from a shared counter once their
// static range is done.  Static ranges keep the partial states few (a unit
// that lies inside one range is finished in place); the dynamic tail evens
// out the finishing times, which otherwise spread by ~20% because some SMs
// get less memory bandwidth than others.
//
// A worker consumes its chunks as one stream: static tiles (its range cut into
// pieces of at most 32 chunks, one descriptor per lane), then dynamic tiles.
// Two tiles are live at a time -- the consumer's and the next one -- and the
// producer (lane 0 issuing the copies) runs at most STAGES chunks ahead, so
// every tile but the very last is at least STAGES chunks long.
//
// Partial-state slots: a segment (the chunks of one unit processed by one
// worker in one piece) of unit u in worker w's static range uses slot u + w;
// one in dynamic tile t uses slot U + NW + u + t (U units, NW workers).  Along
// either region the (u, w) or (u, t) pairs of consecutive segments grow
// monotonically, so these slots never collide.
#pragma once

#include "common.cuh"

namespace pkv {

// One chunk's description, computed by the lane that owns it in a tile.
struct ChunkDesc {
    int u;          // unit = (b * Hkv + h) * sub_groups + sg
    int k;          // chunk index within the unit
    int nch;        // chunks of the unit
    int nvalid;     // valid tokens in the chunk (1..16)
    long long off;  // first pool row of the chunk ([page][h][slot] rows of D), -1: bad page id
};

// Chunk f of the flattened batch.  The sequence holding it is the largest b
// with prefix[b] <= f (empty sequences are skipped); it lies in [lo, hi).
__device__ __forceinline__ ChunkDesc describe_chunk(const DecodeParams& p, int f, int units_per_b,
                                                    int lo, int hi) {
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.prefix + mid) <= f) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int rem = f - __ldg(p.prefix + b);
    const int L = __ldg(p.lens_eff + b);
    const int nch = (L + kChunk - 1) / kChunk;
    const int uidx = rem / nch;
    ChunkDesc d;
    d.k = rem - uidx * nch;
    d.nch = nch;
    d.u = b * units_per_b + uidx;
    d.nvalid = min(kChunk, L - d.k * kChunk);
    const int h = uidx / p.sub_groups;
    const int tok = d.k * kChunk;
    const int page = __ldg(p.table + (long long)b * p.table_stride + tok / p.page_size);
    if (page >= 0 && page < p.num_pages) {
        d.off = (((long long)page * p.n_kv_heads + h) * p.page_size + (tok % p.page_size));
    } else {
        d.off = -1;
        set_status(p.status, PKV_DEV_BAD_PAGE);
    }
    return d;
}

__device__ __forceinline__ ChunkDesc shfl_desc(const ChunkDesc& a, int src) {
    ChunkDesc d;
    d.u = __shfl_sync(kFull, a.u, src);
    d.k = __shfl_sync(kFull, a.k, src);
    d.nch = __shfl_sync(kFull, a.nch, src);
    d.nvalid = __shfl_sync(kFull, a.nvalid, src);
    d.off = __shfl_sync(kFull, a.off, src);
    return d;
}

__device__ __forceinline__ ChunkDesc sel_desc(bool second, const ChunkDesc& a,
                                              const ChunkDesc& b) {
    ChunkDesc d;
    d.u = second ? b.u : a.u;
    d.k = second ? b.k : a.k;
    d.nch = second ? b.nch : a.nch;
    d.nvalid = second ? b.nvalid : a.nvalid;
    d.off = second ? b.off : a.off;
    return d;
}

// The chunk stream of one worker.  All members are warp-uniform except the
// lane-held descriptors wa / wb.  Every method must be called by all 32
// lanes (they shuffle).
struct WorkStream {
    // the live tiles: a = the consumer's, b = the next one (len 0: none yet)
    int a_start, a_len, a_slot, a_contig;
    int b_start, b_len, b_slot, b_contig;
    ChunkDesc wa, wb;
    int stream_end;   // first position past the last chunk (INT_MAX while unknown)
    bool exhausted;   // no tile left to take
    // static range of this worker
    int s_next, s_end, s_tiles_left, s_piece, s_extra;
    int b_lo_static, b_hi_static;
    int lane, gw, units_per_b;

    __device__ __forceinline__ int a_end() const { return a_start + a_len; }

    // Fill tile b (the one after tile a): the next static piece, else a
    // dynamic tile from the shared counter, else mark the stream exhausted.
    __device__ __forceinline__ void acquire(const DecodeParams& p) {
        const int start = a_start + a_len;
        int f, len, slot, contig, lo, hi;
        if (s_tiles_left > 0) {
            len = s_piece + (s_extra > 0 ? 1 : 0);
            s_extra -= (s_extra > 0);
            --s_tiles_left;
            f = s_next;
            s_next += len;
            slot = gw;          // static segment of unit u: slot u + w
            contig = (start > 0);
            lo = b_lo_static;
            hi = b_hi_static;
        } else {
            int t = 0;
            if (lane == 0) t = atomicAdd(p.dyn_next, 1);
            t = __shfl_sync(kFull, t, 0);
            if (t >= p.hdr->dyn_tiles) {
                exhausted = true;
                stream_end = start;
                b_len = 0;
                return;
            }
            const int ts = p.hdr->static_total, K = p.hdr->dyn_tile;
            f = ts + t * K;
            len = min(K, p.hdr->total_chunks - f);
            slot = p.units + p.hdr->num_workers + t;  // dynamic segment: slot U + NW + u + t
            contig = 0;
            lo = __ldg(p.tile_b + t);
            hi = min(p.batch, __ldg(p.tile_b + t + 1) + 1);
        }
        b_start = start;
        b_len = len;
        b_slot = slot;
        b_contig = contig;
        wb.off = -1;
        wb.u = wb.k = wb.nvalid = 0;
        wb.nch = 1;
        if (lane < len) wb = describe_chunk(p, f + lane, units_per_b, lo, hi);
    }

    // Set up the worker's stream; afterwards tile a is its first tile (if any).
    __device__ __forceinline__ void init(const DecodeParams& p, int lane_, int gw_) {
        lane = lane_;
        gw = gw_;
        units_per_b = p.n_kv_heads * p.sub_groups;
        stream_end = 0x7fffffff;
        exhausted = false;
        const int sw = p.hdr->static_per_worker;
        s_next = gw * sw;
        s_end = s_next + sw;
        // cut the static range into pieces of at most 32 chunks, as equal as possible
        s_tiles_left = (sw + 31) / 32;
        s_piece = s_tiles_left ? sw / s_tiles_left : 0;
        s_extra = s_tiles_left ? sw - s_piece * s_tiles_left : 0;
        b_lo_static = __ldg(p.wstart + gw);
        b_hi_static = min(p.batch, __ldg(p.wstart + gw + 1) + 1);
        a_start = 0;
        a_len = 0;
        acquire(p);  // first tile into b, then promote it
        promote();
        if (a_len == 0) stream_end = 0;
    }

    __device__ __forceinline__ void promote() {
        a_start = b_start;
        a_len = b_len;
        a_slot = b_slot;
        a_contig = b_contig;
        wa = wb;
        b_len = 0;
        b_start = a_start + a_len;
    }

    // Consumer at position i: move to the next tile when i leaves tile a, and
    // take the tile after it a few chunks before tile a runs out, so that the
    // producer never waits for it.
    __device__ __forceinline__ void consumer_at(const DecodeParams& p, int i, int lookahead) {
        if (i >= a_end() && b_len > 0) promote();
        if (b_len == 0 && !exhausted && i + lookahead >= a_end()) acquire(p);
    }

    // Producer side: is position j covered by a live tile?  Takes the next
    // tile when none is pending; false for a position past both live tiles
    // (the producer retries after the consumer moved on) or past the end.
    __device__ __forceinline__ bool covered(const DecodeParams& p, int j) {
        if (j < a_end()) return true;
        if (b_len == 0 && !exhausted) acquire(p);
        return b_len > 0 && j < b_start + b_len;
    }

    __device__ __forceinline__ ChunkDesc fetch(int j) const {
        const bool second = j >= a_end();
        const ChunkDesc src = sel_desc(second, wa, wb);
        return shfl_desc(src, j - (second ? b_start : a_start));
    }

    // Partial slot base of position j's tile (slot = base + unit).
    __device__ __forceinline__ int slot_base(int j) const { return j >= a_end() ? b_slot : a_slot; }

    // Does position j (in tile a or b) start a segment?  Does i (in tile a) end one?
    __device__ __forceinline__ bool seg_start(int j, const ChunkDesc& d) const {
        if (d.k == 0) return true;
        if (j == a_start) return !a_contig;
        if (b_len > 0 && j == b_start) return !b_contig;
        return false;
    }
    __device__ __forceinline__ bool seg_end(int i, const ChunkDesc& d) const {
        if (d.k == d.nch - 1 || i + 1 >= stream_end) return true;
        if (i + 1 == a_end()) return !(b_len > 0 && b_contig);
        return false;
    }
};

}  // namespace pkv
