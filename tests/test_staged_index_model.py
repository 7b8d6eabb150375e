"""CPU model of the staged collectives' index arithmetic.

`staged_reduce_kernel` and `staged_copy_kernel` (collectives.cuh) move a tile
of TILE elements per step through a word-major shared-memory tile, with one
global side on vector boundaries and the other shifted by a phase that is
taken in shared memory.  This model restates their index arithmetic (the
`head` skip, the destination `lead`, the source `lag`, the tile reads at an
element shift, the edge elements) on a shrunken block, over random segment
sizes and misalignments for 2- and 4-byte elements and 16- and 32-byte
vectors, and checks that every vector access is aligned and inside its
segment, every element access is in bounds, every shared-memory read is
inside the tile and of a word written in the same step, and the output is the
input.  The CUDA kernels' results are checked against the oracle on the GPU
(odd-shard and random-offset tests); this pins the bounds on the CPU.
"""
import random


def run(kThreads, kStageU, W, EB, n, src_mis, dst_mis, kind, nblocks=3):
    EPV = W * 4 // EB
    VB = 4 * W
    NV = kThreads * kStageU
    TILE = NV * EPV
    KV = NV + 1
    # byte-addressed memories: segment source at src_base, destination at dst_base
    src_base = 4096 + src_mis * EB          # VB-aligned buffer start 4096 plus element offset
    dst_base = 65536 * 8 + dst_mis * EB
    src_vals = [random.getrandbits(8 * EB) for _ in range(n)]
    out = {}
    def load_vec(addr):           # vector load: aligned and fully inside the segment
        assert addr % VB == 0, ("unaligned vector load", addr)
        assert src_base <= addr and addr + VB <= src_base + n * EB, ("vector load outside", addr)
        e = (addr - src_base) // EB
        return [src_vals[e + i] for i in range(EPV)]
    def load_elem(i):
        assert 0 <= i < n, ("element load outside", i)
        return src_vals[i]
    def store_vec(addr, elems):
        assert addr % VB == 0, ("unaligned vector store", addr)
        assert dst_base <= addr and addr + VB <= dst_base + n * EB, ("vector store outside", addr)
        e = (addr - dst_base) // EB
        for i, v in enumerate(elems):
            out[e + i] = v
    def store_elem(i, v):
        assert 0 <= i < n, ("element store outside", i)
        out[i] = v
    def phase(addr):
        return (addr % VB) // EB
    # elements of a vector as word list and back
    def to_words(el):
        if EB == 4:
            return list(el)
        return [el[2 * k] | (el[2 * k + 1] << 16) for k in range(W)]
    def from_words(ws):
        if EB == 4:
            return list(ws)
        r = []
        for w_ in ws:
            r += [w_ & 0xFFFF, w_ >> 16]
        return r
    for_anchor = src_base if kind == "reduce" else dst_base
    head = ((VB - for_anchor % VB) % VB) // EB
    head = min(head, n)
    ntiles = (n - head) // TILE
    for t in range(ntiles):
        e0 = head + t * TILE
        words = [[None] * KV for _ in range(W)]
        def put(v, ws):
            assert 0 <= v < KV
            for k in range(W):
                words[k][v] = ws[k]
        def word(p):
            assert 0 <= p // W < KV, ("smem read outside", p)
            x = words[p % W][p // W]
            assert x is not None, ("smem read of unwritten word", p)
            return x
        def shift(sh):
            # the kernels' StageTile::shift: byte offsets of the W + 1 words
            # that vector 0 reads at element shift sh, and the half-word flag
            ph = sh if EB == 4 else sh >> 1
            at = [(((ph + i) % W) * KV + (ph + i) // W) * 4 for i in range(W + 1)]
            return at, (EB == 2 and sh % 2 == 1)
        def word_at(byte_off):
            j, v = divmod(byte_off // 4, KV)
            assert 0 <= j < W and 0 <= v < KV, ("smem read outside", byte_off)
            x = words[j][v]
            assert x is not None, ("smem read of unwritten word", byte_off)
            return x
        def get_v(v, f):
            at, odd = f
            base = v * 4
            if not odd:
                return [word_at(base + at[k]) for k in range(W)]
            lo = word_at(base + at[0]); r = []
            for k in range(W):
                hi = word_at(base + at[k + 1])
                r.append(((lo >> 16) | (hi << 16)) & 0xFFFFFFFF)
                lo = hi
            return r
        def elem(e):
            if EB == 4:
                return word(e)
            return (word(e >> 1) >> (16 * (e & 1))) & 0xFFFF
        if kind == "reduce":
            for slot in range(NV):
                el = load_vec(src_base + (e0 + slot * EPV) * EB)
                put(slot, to_words(el))
            lead = (EPV - phase(dst_base + e0 * EB)) % EPV
            nvec = (TILE - lead) // EPV
            f = shift(lead)
            for k in range(nvec):
                off = lead + k * EPV
                store_vec(dst_base + (e0 + off) * EB, from_words(get_v(k, f)))
            tail0 = lead + nvec * EPV
            for e in range(lead + (TILE - tail0)):
                te = e if e < lead else tail0 + (e - lead)
                store_elem(e0 + te, elem(te))
        else:
            lag = phase(src_base + e0 * EB)
            nsv = NV + (1 if lag else 0)
            for j in range(nsv):
                s0 = e0 - lag + j * EPV
                if s0 >= 0 and s0 + EPV <= n:
                    el = load_vec(src_base + s0 * EB)
                else:
                    el = [load_elem(s0 + e) if 0 <= s0 + e < n else 0 for e in range(EPV)]
                put(j, to_words(el))
            f = shift(lag)
            for k in range(NV):
                store_vec(dst_base + (e0 + k * EPV) * EB, from_words(get_v(k, f)))
    # scalar ranges
    for i in list(range(0, head)) + list(range(head + ntiles * TILE, n)):
        store_elem(i, load_elem(i))
    assert len(out) == n and all(out[i] == src_vals[i] for i in range(n)), "wrong result"



def test_staged_index_arithmetic_random_segments():
    rng_state = random.getstate()
    random.seed(1)
    try:
        for _ in range(6000):
            kThreads = random.choice([2, 3, 4])
            kStageU = random.choice([1, 2])
            W = random.choice([4, 8])
            EB = random.choice([2, 4])
            EPV = W * 4 // EB
            kind = random.choice(["reduce", "copy"])
            n = random.randint(0, 5 * kThreads * kStageU * EPV + 7)
            src_mis = random.randint(0, EPV - 1)
            dst_mis = random.randint(0, EPV - 1)
            run(kThreads, kStageU, W, EB, n, src_mis, dst_mis, kind)
    finally:
        random.setstate(rng_state)
