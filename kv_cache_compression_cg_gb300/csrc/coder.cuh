// coder.cuh - range-encoder state and steps shared by the slice coders
// (specification R of include/cachegen.h).
//
// State lives in registers: 32-bit low/range plus a 64-bit accumulator of
// emitted-but-unwritten bits, so a carry is a plain add into the accumulator;
// full words leave it one behind ("prev"), so only a carry through 32 or more
// one-bits ever touches stored bytes again.
#pragma once

#include <cstdint>

#include "cg_internal.cuh"

namespace cg {
namespace {

struct Enc {
    uint32_t low, range;
    uint32_t alo, ahi;  // 64-bit accumulator of pending output bits [0, nbits),
                        // plus a carry at bit nbits
    uint32_t nbits;     // multiple of 8
    uint32_t prev;      // last full word, not yet stored (absorbs carries)
    int npush;          // words pushed so far; word i is stored at index i - 1
};

__device__ __forceinline__ void enc_init(Enc &e) {
    e.low = 0;
    e.range = 0xFFFFFFFFu;
    e.alo = 0;
    e.ahi = 0;
    e.nbits = 0;
    e.prev = 0;
    e.npush = 0;
}

// Add one to the bytes [0, nbytes) already stored (the carry rule).
__device__ __noinline__ void carry_into_stored(uint8_t *stream, int nbytes) {
    int i = nbytes - 1;
    while (i >= 0 && stream[i] == 0xFF) {
        stream[i] = 0;
        i--;
    }
    if (i >= 0) stream[i] = (uint8_t)(stream[i] + 1);
}

__device__ __forceinline__ void store_be(uint8_t *stream, int idx, uint32_t w) {
    reinterpret_cast<uint32_t *>(stream)[idx] = __byte_perm(w, 0, 0x0123);
}

// Hand the pending word over: the carry goes into it (and, if it wraps, into
// the stored bytes), it is stored at index npush - 1 (the first push parks the
// empty placeholder in the slack before the stream), and `word` becomes the
// pending one.
__device__ __forceinline__ void enc_push_word(Enc &e, uint8_t *stream, uint32_t word, uint32_t ovf) {
    e.prev += ovf;
    if (ovf != 0u && e.prev == 0u) carry_into_stored(stream, 4 * (e.npush - 1));
    store_be(stream, e.npush - 1, e.prev);
    e.npush++;
    e.prev = word;
}

// Move the oldest 32 pending bits out of the accumulator (needs nbits >= 32).
__device__ __forceinline__ void enc_flush_word(Enc &e, uint8_t *stream) {
    const uint32_t k = e.nbits - 32;  // bits left after this word, < 32
    uint32_t word, ovf, mask;
    asm("shf.r.clamp.b32 %0, %1, %2, %3;" : "=r"(word) : "r"(e.alo), "r"(e.ahi), "r"(k));
    ovf = (e.ahi >> k) & 1u;
    asm("bmsk.clamp.b32 %0, 0, %1;" : "=r"(mask) : "r"(k));
    e.alo &= mask;
    e.ahi = 0;
    e.nbits = k;
    enc_push_word(e, stream, word, ovf);
}

// Code one symbol given its packed CDF entry (lo | f << 16): r = range >> 16;
// low += r*lo with the carry going into the accumulator; range = r*f; then
// shift out 0, 1 or 2 bytes (clz(range) & 24 bits) from low into the
// accumulator.
__device__ __forceinline__ void enc_symbol(Enc &e, uint32_t entry) {
    asm("{\n\t"
        ".reg .u32 r, lo, f, sh;\n\t"
        "shr.b32 r, %1, 16;\n\t"
        "and.b32 lo, %5, 65535;\n\t"
        "shr.b32 f, %5, 16;\n\t"
        "mad.lo.cc.u32 %0, r, lo, %0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.u32 %3, %3, 0;\n\t"
        "mul.lo.u32 %1, r, f;\n\t"
        "clz.b32 sh, %1;\n\t"
        "and.b32 sh, sh, 24;\n\t"
        "shf.l.clamp.b32 %3, %2, %3, sh;\n\t"
        "shf.l.clamp.b32 %2, %0, %2, sh;\n\t"
        "shl.b32 %0, %0, sh;\n\t"
        "shl.b32 %1, %1, sh;\n\t"
        "add.u32 %4, %4, sh;\n\t"
        "}"
        : "+r"(e.low), "+r"(e.range), "+r"(e.alo), "+r"(e.ahi), "+r"(e.nbits)
        : "r"(entry));
}

// The same step with the CDF entry already split into lo and f.
__device__ __forceinline__ void enc_symbol_lf(Enc &e, uint32_t lo, uint32_t f) {
    asm("{\n\t"
        ".reg .u32 r, sh;\n\t"
        "shr.b32 r, %1, 16;\n\t"
        "mad.lo.cc.u32 %0, r, %5, %0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.u32 %3, %3, 0;\n\t"
        "mul.lo.u32 %1, r, %6;\n\t"
        "clz.b32 sh, %1;\n\t"
        "and.b32 sh, sh, 24;\n\t"
        "shf.l.clamp.b32 %3, %2, %3, sh;\n\t"
        "shf.l.clamp.b32 %2, %0, %2, sh;\n\t"
        "shl.b32 %0, %0, sh;\n\t"
        "shl.b32 %1, %1, sh;\n\t"
        "add.u32 %4, %4, sh;\n\t"
        "}"
        : "+r"(e.low), "+r"(e.range), "+r"(e.alo), "+r"(e.ahi), "+r"(e.nbits)
        : "r"(lo), "r"(f));
}

// The same step with the entry packed as lo | (f - 1) << 16, which holds every
// f up to 65536: range = r (f - 1) + r.
__device__ __forceinline__ void enc_symbol_m1(Enc &e, uint32_t entry) {
    asm("{\n\t"
        ".reg .u32 r, lo, fm, sh;\n\t"
        "shr.b32 r, %1, 16;\n\t"
        "and.b32 lo, %5, 65535;\n\t"
        "shr.b32 fm, %5, 16;\n\t"
        "mad.lo.cc.u32 %0, r, lo, %0;\n\t"
        "addc.cc.u32 %2, %2, 0;\n\t"
        "addc.u32 %3, %3, 0;\n\t"
        "mad.lo.u32 %1, r, fm, r;\n\t"
        "clz.b32 sh, %1;\n\t"
        "and.b32 sh, sh, 24;\n\t"
        "shf.l.clamp.b32 %3, %2, %3, sh;\n\t"
        "shf.l.clamp.b32 %2, %0, %2, sh;\n\t"
        "shl.b32 %0, %0, sh;\n\t"
        "shl.b32 %1, %1, sh;\n\t"
        "add.u32 %4, %4, sh;\n\t"
        "}"
        : "+r"(e.low), "+r"(e.range), "+r"(e.alo), "+r"(e.ahi), "+r"(e.nbits)
        : "r"(entry));
}

// enc_flush_word when nbits >= 32, without a branch, for the latency-mode
// coders, where each stream's dependent chain sets the time: the word's store
// is predicated and the state updates are selects; only a carry out of the
// pending word (rare) branches, to the stored bytes. The throughput coder keeps
// the branch (there every unconditional instruction costs issue slots).
__device__ __forceinline__ void enc_flush_sel(Enc &e, uint8_t *stream) {
    const bool need = e.nbits >= 32;
    const uint32_t k = need ? e.nbits - 32 : 0u;  // bits left after the word
    uint32_t word, mask;
    asm("shf.r.clamp.b32 %0, %1, %2, %3;" : "=r"(word) : "r"(e.alo), "r"(e.ahi), "r"(k));
    const uint32_t ovf = need ? (e.ahi >> k) & 1u : 0u;
    asm("bmsk.clamp.b32 %0, 0, %1;" : "=r"(mask) : "r"(k));
    e.alo = need ? (e.alo & mask) : e.alo;
    e.ahi = need ? 0u : e.ahi;
    e.nbits = need ? k : e.nbits;
    // enc_push_word's steps, predicated
    const uint32_t pv = e.prev + ovf;
    if (ovf != 0u && pv == 0u) carry_into_stored(stream, 4 * (e.npush - 1));
    if (need) store_be(stream, e.npush - 1, pv);
    e.npush += need ? 1 : 0;
    e.prev = need ? word : e.prev;
}

// Flush byte and final words; returns the stream length in bytes.
__device__ __forceinline__ uint32_t enc_finish(Enc &e, uint8_t *stream) {
    if (e.nbits >= 32) enc_flush_word(e, stream);
    // flush byte: v = low + 0x00FFFFFF (carry into the accumulator), emit v >> 24
    const uint32_t v = e.low + 0x00FFFFFFu;
    const uint32_t c = v < e.low ? 1u : 0u;
    asm("add.cc.u32 %0, %0, %2;\n\taddc.u32 %1, %1, 0;" : "+r"(e.alo), "+r"(e.ahi) : "r"(c));
    asm("shf.l.clamp.b32 %0, %1, %0, 8;" : "+r"(e.ahi) : "r"(e.alo));
    e.alo = (e.alo << 8) | (v >> 24);
    e.nbits += 8;
    if (e.nbits >= 32) enc_flush_word(e, stream);
    // now nbits < 32: pending bits and the carry bit both sit in alo
    const uint32_t ovf = (e.alo >> e.nbits) & 1u;
    if (e.npush > 0) {  // the pending word is real: apply the carry, store it
        e.prev += ovf;
        if (ovf != 0u && e.prev == 0u) carry_into_stored(stream, 4 * (e.npush - 1));
        store_be(stream, e.npush - 1, e.prev);
    }
    if (e.nbits > 0) {
        uint32_t mask;
        asm("bmsk.clamp.b32 %0, 0, %1;" : "=r"(mask) : "r"(e.nbits));
        store_be(stream, e.npush, (e.alo & mask) << (32 - e.nbits));
    }
    return (uint32_t)(4 * e.npush + e.nbits / 8);
}

}  // namespace
}  // namespace cg
