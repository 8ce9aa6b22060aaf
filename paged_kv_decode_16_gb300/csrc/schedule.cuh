// schedule.cuh -- which 16-token chunks each decode worker (one warp) handles.
//
// All chunks of the batch are laid end to end: sequence-major, then KV head
// (and query sub-group), then chunk.  That order is cut into one contiguous
// range per worker, as equal as possible: with T chunks and NW workers,
// sw = T / NW and r = T % NW, workers 0 .. r-1 take sw + 1 chunks and the
// others sw.  Every warp gets the same work to within one chunk, whatever the
// length mix, and a unit (sequence, KV head, sub-group) that lies inside one
// range is finished in place.
//
// A worker consumes its range as a stream of tiles of at most 32 chunks (one
// descriptor per lane, as equal as possible).  Two tiles are live at a time --
// the consumer's and the next one -- and the producer (lane 0 issuing the
// copies) runs at most STAGES chunks ahead.
//
// Partial-state slots: the segment (chunks of one unit in one worker's range)
// of unit u in worker w's range uses slot u + w.  Along the order the (u, w)
// pairs of consecutive segments grow monotonically, so slots never collide;
// there are at most U + NW of them.  A range holds at most two segments that
// are not a whole unit: its first and its last.
#pragma once

#include "common.cuh"

namespace pkv {

// One chunk's description, computed by the lane that owns it in a tile.
struct ChunkDesc {
    int u;          // unit = (b * Hkv + h) * sub_groups + sg
    int k;          // chunk index within the unit
    int nch;        // chunks of the unit
    int nvalid;     // valid tokens in the chunk (1..16)
    int len;        // tokens of the sequence
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
    d.len = L;
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
    d.len = __shfl_sync(kFull, a.len, src);
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
    d.len = second ? b.len : a.len;
    d.off = second ? b.off : a.off;
    return d;
}

// The chunk stream of one worker.  All members are warp-uniform except the
// lane-held descriptors wa / wb.  Every method must be called by all 32
// lanes (they shuffle).
struct WorkStream {
    // the live tiles: a = the consumer's, b = the next one (len 0: none yet)
    int a_start, a_len;
    int b_start, b_len;
    ChunkDesc wa, wb;
    int stream_end;   // chunks in this worker's range
    // the rest of the range: next chunk, tiles left, base tile length, longer tiles
    int next_f, tiles_left, piece, extra;
    int b_lo, b_hi;   // sequences of the range: [b_lo, b_hi)
    int lane, gw, units_per_b, slot_base;
    int range_f0, sw, r;  // first chunk of the range; the split (chunks_per_worker, extra)

    __device__ __forceinline__ int a_end() const { return a_start + a_len; }

    // Fill tile b (the one after tile a) with the next piece of the range.
    __device__ __forceinline__ void acquire(const DecodeParams& p) {
        b_start = a_start + a_len;
        b_len = 0;
        if (tiles_left == 0) return;
        const int len = piece + (extra > 0 ? 1 : 0);
        extra -= (extra > 0);
        --tiles_left;
        const int f = next_f;
        next_f += len;
        b_len = len;
        wb.off = -1;
        wb.u = wb.k = wb.nvalid = wb.len = 0;
        wb.nch = 1;
        if (lane < len) wb = describe_chunk(p, f + lane, units_per_b, b_lo, b_hi);
    }

    // Set up the worker's stream; afterwards tile a is its first tile (if any).
    __device__ __forceinline__ void init(const DecodeParams& p, int lane_, int gw_) {
        lane = lane_;
        gw = gw_;
        units_per_b = p.n_kv_heads * p.sub_groups;
        slot_base = gw;  // segment of unit u in this range: slot u + w
        sw = p.hdr->chunks_per_worker;
        r = p.hdr->extra_chunks;
        range_f0 = range_begin(gw, sw, r);
        next_f = range_f0;
        stream_end = sw + (gw < r ? 1 : 0);
        // cut the range into tiles of at most 32 chunks, as equal as possible
        tiles_left = (stream_end + 31) / 32;
        piece = tiles_left ? stream_end / tiles_left : 0;
        extra = tiles_left ? stream_end - piece * tiles_left : 0;
        b_lo = __ldg(p.wstart + gw);
        b_hi = min(p.batch, __ldg(p.wstart + gw + 1) + 1);
        a_start = 0;
        a_len = 0;
        acquire(p);  // first tile into b, then promote it
        promote();
    }

    __device__ __forceinline__ void promote() {
        a_start = b_start;
        a_len = b_len;
        wa = wb;
        b_len = 0;
        b_start = a_start + a_len;
    }

    // Consumer at position i: move to the next tile when i leaves tile a, and
    // take the tile after it a few chunks before tile a runs out, so that the
    // producer never waits for it.
    __device__ __forceinline__ void consumer_at(const DecodeParams& p, int i, int lookahead) {
        if (i >= a_end() && b_len > 0) promote();
        if (b_len == 0 && tiles_left > 0 && i + lookahead >= a_end()) acquire(p);
    }

    // Producer side: is position j covered by a live tile?  Takes the next
    // tile when none is pending; false for a position past both live tiles
    // (the producer retries after the consumer moved on) or past the end.
    __device__ __forceinline__ bool covered(const DecodeParams& p, int j) {
        if (j < a_end()) return true;
        if (j >= stream_end) return false;
        if (b_len == 0 && tiles_left > 0) acquire(p);
        return b_len > 0 && j < b_start + b_len;
    }

    __device__ __forceinline__ ChunkDesc fetch(int j) const {
        const bool second = j >= a_end();
        const ChunkDesc src = sel_desc(second, wa, wb);
        return shfl_desc(src, j - (second ? b_start : a_start));
    }

    // Does position j start a segment (a unit's first chunk, or the range's
    // first)?  Does position i end one (a unit's last chunk, or the range's
    // last)?
    __device__ __forceinline__ bool seg_start(int j, const ChunkDesc& d) const {
        return d.k == 0 || j == 0;
    }
    __device__ __forceinline__ bool seg_end(int i, const ChunkDesc& d) const {
        return d.k == d.nch - 1 || i + 1 >= stream_end;
    }
};

}  // namespace pkv
