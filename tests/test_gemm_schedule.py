"""Host-side check of the GEMM's work schedule (no GPU).

The kernel's per-CTA work walk (data-parallel waves, then stream-K over the
remaining tiles, fixed by the same integer formulas in the producer, MMA and
epilogue roles) is mirrored here and checked for every workload shape:
every (tile, K block) iteration is covered exactly once, every CTA's
stream-K range is non-empty, the parts of each split tile are numbered
0..nparts-1 by consecutive CTAs, and the partial slots they use are
distinct. A mistake here would leave an output tile unwritten or let two
CTAs race on one slot."""
import itertools
import os
import shutil
import subprocess

import pytest


MAX_COUNTERS = 64 * 1024 // 4   # the workspace's fixed counter region, one int32 per tile


def make_plan(M, N, K, sms, pairs=None, split_k=True):
    """pairs: co-resident CTA pairs of the cluster kernel (default sms // 2;
    0 disables clusters). With pairs, large-M tiles of 128 x 256 run as
    cluster pairs: the schedule's lane index counts pairs of 128-row tiles.
    split_k=False: no split-K clusters (their capacity is unknown, as when
    the library plans without a device)."""
    if pairs is None:
        pairs = sms // 2
    Kb = K // 128
    if M <= 128:
        swap = True
        bn = 16 if M <= 16 else 32 if M <= 32 else 64 if M <= 64 else 128
        tl, tc = -(-N // 128), -(-M // bn)
        tiles = tl * tc
        if 2 * tiles >= sms:   # decode (any token-tile width): whole weight tiles
            if tiles <= sms:                 # one CTA per tile
                return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=tiles, dp=1, sk_tiles=0, sk_iters=0, Kb=Kb,
                            tiles=tiles, cluster=1, ksplit=1)
            return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=sms, dp=0, sk_tiles=0, sk_iters=0, Kb=Kb,
                        tiles=tiles, cluster=1, ksplit=1, whole=tiles)   # round-robin beyond one per SM
        if split_k and 2 * tiles < sms:   # few tiles: split-K clusters of ks CTAs per tile
            for ks in (8, 4, 2):      # (co-resident clusters assumed: sms // ks)
                if Kb >= 2 * ks and tiles * ks <= sms:
                    return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=tiles * ks, dp=1, sk_tiles=0, sk_iters=0,
                                Kb=Kb, tiles=tiles, cluster=1, ksplit=ks)
    else:
        swap = False
        tiles256 = -(-M // 128) * -(-N // 256)
        bn = 128 if (N <= 128 or Kb <= 4 or tiles256 < 2 * sms) else 256
        tl, tc = -(-M // 128), -(-N // bn)
    cluster = 1
    workers = sms
    if not swap and bn == 256 and pairs > 0:
        cluster, workers = 2, pairs
        tl = (tl + 1) // 2
    tiles = tl * tc
    rounds = -(-tiles // workers)
    if not swap and tiles * cluster <= MAX_COUNTERS and rounds * Kb * workers - tiles * Kb <= 32 * workers:
        # dense large-M tiles: whole tiles unless stream-K saves the busiest worker more than 32 K blocks
        return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=min(tiles, workers), dp=0, sk_tiles=0, sk_iters=0, Kb=Kb,
                    tiles=tiles, cluster=cluster, ksplit=1, whole=tiles)
    if tiles * cluster > MAX_COUNTERS:   # more tiles than the counter region holds: whole tiles only
        return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=workers, dp=0, sk_tiles=0, sk_iters=0, Kb=Kb,
                    tiles=tiles, cluster=cluster, ksplit=1, whole=tiles)
    if tiles >= 2 * workers:
        grid = workers
        dp = tiles // workers - 1
        sk_tiles = tiles - dp * workers
    else:
        dp = 0
        sk_tiles = tiles
        grid = min(workers, tiles * Kb)
    return dict(swap=swap, bn=bn, tl=tl, tc=tc, grid=grid, dp=dp, sk_tiles=sk_tiles,
                sk_iters=sk_tiles * Kb, Kb=Kb, tiles=tiles, cluster=cluster, ksplit=1)


def units(p, c):
    if p["ksplit"] > 1:      # CTA c: tile c // ks, K slice c % ks (mirror of the split-K branch)
        ks, Kb = p["ksplit"], p["Kb"]
        r = c % ks
        yield (c // ks, r * Kb // ks, (r + 1) * Kb // ks, 0, 1)
        return
    G, Kb, S = p["grid"], p["Kb"], p["sk_iters"]
    if p.get("whole"):       # round-robin whole tiles (mirror of the whole_tiles branch)
        for t in range(c, p["whole"], G):
            yield (t, 0, Kb, 0, 1)
        return
    for j in range(p["dp"]):
        yield (c + j * G, 0, Kb, 0, 1)
    it, it_end = c * S // G, (c + 1) * S // G

    def cta_of(i):
        return ((i + 1) * G - 1) // S

    while it < it_end:
        t = it // Kb
        tb, te = t * Kb, t * Kb + Kb
        seg = min(te, it_end)
        first, last = cta_of(tb), cta_of(te - 1)
        yield (p["dp"] * G + t, it - tb, seg - tb, c - first, last - first + 1)
        it = seg


SHAPES = [
    (16, 320, 256), (1, 10944, 2048), (8, 10944, 2048), (64, 10944, 2048),
    (4096, 18432, 7168), (4096, 7168, 18432),
    (64, 1536, 7168), (64, 576, 7168), (64, 24576, 1536), (64, 32768, 512), (8, 65536, 1024), (32, 40960, 1536),
    (2048, 1536, 7168), (2048, 576, 7168), (2048, 24576, 1536), (2048, 32768, 512),
    (129, 130, 128), (300, 700, 384), (1, 1, 128), (128, 129, 2048), (33, 4000, 128),
    (5000, 100, 256),
    (40000, 60000, 256),   # more tiles than counters: whole tiles, round-robin
]


@pytest.mark.parametrize("sms", [152, 148, 7])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_schedule_covers_every_iteration_once(M, N, K, sms):
    p = make_plan(M, N, K, sms)
    G, Kb = p["grid"], p["Kb"]
    assert G >= 1 and p["sk_iters"] >= G or p["sk_iters"] == 0
    cover = {}
    slots = {}
    parts = {}
    for c in range(G):
        S = p["sk_iters"]
        if S:
            assert (c + 1) * S // G > c * S // G, "empty stream-K range"
        for tile, kb0, kb1, part, nparts in units(p, c):
            assert 0 <= tile < p["tiles"] and 0 <= kb0 < kb1 <= Kb
            for kb in range(kb0, kb1):
                assert (tile, kb) not in cover
                cover[(tile, kb)] = c
            if nparts > 1:
                assert 0 <= part < nparts
                slot = 2 * c + (1 if part == 0 else 0)
                assert slot not in slots, "two partials in one slot"
                slots[slot] = (tile, part)
                parts.setdefault(tile, {})[part] = (c, kb0, kb1)
            elif p["ksplit"] == 1:
                assert kb0 == 0 and kb1 == Kb
    assert len(cover) == p["tiles"] * Kb
    for tile, ps in parts.items():
        n = len(ps)
        assert sorted(ps) == list(range(n))
        cs = [ps[i][0] for i in range(n)]
        assert cs == list(range(cs[0], cs[0] + n)), "parts come from consecutive CTAs"
        # the parts tile the K range in order
        assert ps[0][1] == 0 and ps[n - 1][2] == Kb
        for i in range(n - 1):
            assert ps[i][2] == ps[i + 1][1]
        # the reducer finds each part's slot from (first CTA, part index)
        for i in range(n):
            assert slots[2 * (cs[0] + i) + (1 if i == 0 else 0)] == (tile, i)


@pytest.mark.parametrize("M,N,K", [(64, 1536, 7168), (64, 576, 7168), (8, 1536, 7168), (50, 300, 1024),
                                   (1, 640, 4096), (100, 1536, 512), (17, 576, 7168)])
def test_split_k_clusters(M, N, K):
    """Few weight tiles: clusters of ks CTAs per tile, every CTA a non-empty K
    slice, and the reduction's column slices (BN / ks per rank) cover the tile."""
    p = make_plan(M, N, K, 152)
    ks = p["ksplit"]
    assert ks in (2, 4, 8) and p["grid"] == p["tiles"] * ks and p["grid"] <= 152
    assert p["bn"] % ks == 0
    per = p["bn"] // ks
    cols = sorted(r * per + j for r in range(ks) for j in range(per))
    assert cols == list(range(p["bn"]))
    for t in range(p["tiles"]):
        slices = [u for c in range(t * ks, (t + 1) * ks) for u in units(p, c)]
        assert all(u[0] == t and u[2] - u[1] >= 2 for u in slices)
        assert sorted((u[1], u[2]) for u in slices)[0][0] == 0 and max(u[2] for u in slices) == p["Kb"]


def test_decode_plan_uses_whole_tiles():
    p = make_plan(8, 10944, 2048, 152)
    assert p["swap"] and p["bn"] == 16 and p["grid"] == 86 and p["dp"] == 1 and p["sk_iters"] == 0
    p = make_plan(64, 10944, 2048, 152)      # BN 64: whole tiles as well
    assert p["bn"] == 64 and p["grid"] == 86 and p["dp"] == 1
    p = make_plan(128, 10944, 2048, 152)     # BN 128: whole tiles as well
    assert p["bn"] == 128 and p["grid"] == 86 and p["dp"] == 1
    p = make_plan(128, 3000, 2048, 152)      # few tiles: split-K clusters
    assert p["ksplit"] == 4 and p["grid"] == 96
    p = make_plan(128, 3000, 2048, 152, split_k=False)   # ... or, without them, stream-K
    assert p["grid"] == 152 and p["dp"] == 0 and p["sk_tiles"] == 24
    p = make_plan(8, 24576, 1536, 152)       # 192 tiles: whole tiles, round-robin over every SM
    assert p["grid"] == 152 and p["whole"] == 192 and p["sk_iters"] == 0
    assert [u[0] for u in units(p, 3)] == [3, 155] and [u[0] for u in units(p, 40)] == [40]


def test_tile_width_rule():
    """128-column tiles where 128 x 256 tiles would number fewer than two per
    SM or K <= 512; 128 x 256 cluster pairs for the large prefill shapes."""
    for M, N, K in [(2048, 1536, 7168), (2048, 576, 7168), (2048, 32768, 512), (300, 576, 1024)]:
        assert make_plan(M, N, K, 152)["bn"] == 128
    for M, N, K in [(4096, 18432, 7168), (4096, 7168, 18432), (2048, 24576, 1536), (1300, 7000, 640)]:
        p = make_plan(M, N, K, 152)
        assert p["bn"] == 256 and p["cluster"] == 2


def test_prefill_plan_is_hybrid():
    p = make_plan(4096, 18432, 7168, 152, pairs=0)
    assert not p["swap"] and p["bn"] == 256 and p["dp"] == 14 and p["sk_tiles"] == 2304 - 14 * 152
    # cluster pairs: 16 pair rows x 72 column tiles over 76 pairs
    p = make_plan(4096, 18432, 7168, 152)
    assert p["cluster"] == 2 and p["tl"] == 16 and p["grid"] == 76 and p["dp"] == 14
    assert p["sk_tiles"] == 1152 - 14 * 76


def tile_of(p, tile, rank):
    """Mirror of the kernel's (schedule tile, cluster rank) -> (128-row lane tile,
    column tile, counter index)."""
    tl = (tile % p["tl"]) * p["cluster"] + rank
    tc = tile // p["tl"]
    return tl, tc, tile * p["cluster"] + rank


# (SM counts chosen so that each shape takes 128 x 256 tiles in cluster pairs:
# at least two such tiles per SM, K > 512.)
@pytest.mark.parametrize("M,N,K,sms", [(4096, 18432, 7168, 152), (300, 700, 640, 4), (129, 300, 1024, 2),
                                       (2048, 576, 7168, 16), (5000, 1000, 640, 64), (1300, 7000, 640, 152)])
def test_cluster_pairs_cover_every_output_tile_once(M, N, K, sms):
    p = make_plan(M, N, K, sms)
    assert p["cluster"] == 2
    m_tiles, n_tiles = -(-M // 128), -(-N // 256)
    seen, counters = set(), set()
    for tile in range(p["tiles"]):
        for rank in range(2):
            tl, tc, ctr = tile_of(p, tile, rank)
            assert ctr not in counters and 0 <= ctr < p["tiles"] * 2
            counters.add(ctr)
            if tl < m_tiles:            # the second CTA of the last pair may own no rows
                assert (tl, tc) not in seen
                seen.add((tl, tc))
            else:
                assert tl == m_tiles and m_tiles % 2 == 1
    assert seen == {(a, b) for a in range(m_tiles) for b in range(n_tiles)}


def test_cluster_pair_slots_are_distinct():
    """Stream-K partial slots: CTA (worker w, rank r) owns slots 2 (2 w + r) and
    2 (2 w + r) + 1; the reducer of part q reads worker first + q, same rank."""
    p = make_plan(4096, 7168, 18432, 152)
    G = p["grid"]
    owners = {}
    for w in range(G):
        for r in range(2):
            for k in range(2):
                s = 2 * (2 * w + r) + k
                assert s not in owners
                owners[s] = (w, r)
    assert len(owners) == 4 * G


# ---- grouped (per-expert) tiles and the routing permutation -------------------

def grouped_tile(tile, mtiles, tiles_col, E):
    """Mirror of the kernel's tile -> (group, column tile, row tile) mapping."""
    lo, hi = 0, E - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if mtiles[mid] * tiles_col <= tile:
            lo = mid
        else:
            hi = mid - 1
    e = lo
    mt_e = mtiles[e + 1] - mtiles[e]
    local = tile - mtiles[e] * tiles_col
    return e, local // mt_e, local % mt_e


@pytest.mark.parametrize("seed", range(6))
def test_grouped_tiles_cover_every_group_tile_once(seed):
    import numpy as np

    g = np.random.Generator(np.random.PCG64(seed))
    E = int(g.integers(1, 40))
    counts = g.integers(0, 400, E) * (g.random(E) < 0.7)       # some empty experts
    mt = -(-counts // 128)
    mtiles = np.concatenate([[0], np.cumsum(mt)])
    tiles_col = int(g.integers(1, 30))
    want = {(e, nt, m) for e in range(E) for nt in range(tiles_col) for m in range(mt[e])}
    got = [grouped_tile(t, mtiles, tiles_col, E) for t in range(int(mtiles[-1]) * tiles_col)]
    assert len(got) == len(set(got)) and set(got) == want


def permute_mirror(idx, E, chunk=1024):
    """Mirror of the three-pass permutation. Rank pass, per chunk of pairs:
    a pair's rank is its rank among its warp's earlier pairs of the same
    expert plus that expert's count in the chunk's earlier warps, and the
    chunk's histogram. Offsets pass: per-(chunk, expert) bases. Scatter pass:
    perm[base + rank] = pair."""
    import numpy as np

    flat = idx.ravel()
    n = flat.size
    nchunks = -(-n // chunk)
    rank = np.full(n, -1)
    hist = np.zeros((nchunks, E), np.int64)
    for c in range(nchunks):
        c0 = c * chunk
        wtab = np.zeros((chunk // 32, E), np.int64)
        wrank = {}
        for i in range(c0, min(c0 + chunk, n)):
            e = flat[i]
            if not (0 <= e < E):
                continue
            w = (i - c0) // 32
            wrank[i] = sum(1 for j in range(c0 + w * 32, i) if flat[j] == e)
            wtab[w, e] += 1
        for i, r in wrank.items():
            w = (i - c0) // 32
            rank[i] = wtab[:w, flat[i]].sum() + r
        hist[c] = wtab.sum(axis=0)
    counts = hist.sum(axis=0)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    base = offsets[:-1][None, :] + np.cumsum(hist, axis=0) - hist
    perm = np.full(n, -1)
    for i in range(n):
        e = flat[i]
        if 0 <= e < E:
            perm[base[i // chunk, e] + rank[i]] = i
    return counts, offsets, perm[: offsets[-1]]


def test_permute_mirror_is_the_stable_sort():
    import numpy as np

    import oracle
    import synthetic

    idx, _ = synthetic.moe_routing(300, 16, 4, 91, zipf_s=1.2)
    c, o, p = permute_mirror(idx, 16, chunk=256)
    co, oo, po = oracle.moe_permute(idx, 16)
    assert np.array_equal(c, co) and np.array_equal(o, oo) and np.array_equal(p, po)
    bad = idx.copy()
    bad[3, 1] = 99
    bad[7, 0] = -1
    c, o, p = permute_mirror(bad, 16, chunk=256)
    keep = np.flatnonzero((bad.ravel() >= 0) & (bad.ravel() < 16))
    assert np.array_equal(p, keep[np.argsort(bad.ravel()[keep], kind="stable")])


def test_dense_plans_prefer_whole_tiles():
    """Large-M tiles run whole (round-robin over SMs or CTA pairs) unless
    stream-K shortens the busiest worker by more than 32 K blocks."""
    whole = [(2048, 576, 7168), (512, 7168, 2048), (256, 18432, 7168), (4096, 7168, 18432), (1300, 7000, 640)]
    streamk = [(2048, 1536, 7168), (4096, 18432, 7168)]
    for M, N, K in whole:
        p = make_plan(M, N, K, 152)
        assert p.get("whole") == p["tiles"] and p["sk_iters"] == 0, (M, N, K)
    for M, N, K in streamk:
        p = make_plan(M, N, K, 152)
        assert not p.get("whole") and p["sk_tiles"] > 0, (M, N, K)


# ---- the slice-per-SM decode kernel (M <= 16) -------------------------------------

DECODE_SMEM_LIMIT = 232448


def decode_plan(M, N, K, sms, boxes=4, target_warps=16):
    """Mirror of the decode kernel's plan: one CTA per slice of R weight rows
    (ceil(N / SMs) rounded up to 8), the slice in `boxes` TMA boxes of kbb K
    blocks, warps = K slices x row-group parts (at most 5 groups of 16 rows
    per warp with one token fragment, 3 with two). None where the kernel does
    not take the shape (then the tcgen05 swapped kernel runs)."""
    if not 1 <= M <= 16 or N < 1 or K < 128 or K % 128:
        return None
    Kb = K // 128
    R = -(-N // sms)
    R = -(-R // 8) * 8
    if R > 256:
        return None
    nbox = min(Kb, boxes)
    kbb = -(-Kb // nbox)
    if kbb > 256:
        return None
    nbox = -(-Kb // kbb)
    groups = -(-R // 16)
    nt = 1 if M <= 8 else 2
    gpw = 5 if nt == 1 else 3
    gparts = -(-groups // gpw)
    ks = min(max(1, target_warps // gparts), Kb)
    more = target_warps // ks
    if more > gparts:
        gparts = min(more, groups)
    tok = 8 * nt
    wbytes = nbox * kbb * R * 128
    pbytes = ks * tok * (groups * 16 + 4) * 4
    area = -(-max(wbytes, pbytes) // 16) * 16
    wblk = (R + 127) // 128 + 1
    off_bar = -(-(area + wblk * Kb * 4) // 8) * 8
    smem = 1024 + off_bar + nbox * 8 + 8
    if smem > DECODE_SMEM_LIMIT or ks * gparts > 16:
        return None
    return dict(R=R, ctas=-(-N // R), groups=groups, ks=ks, gparts=gparts, gpw=gpw, warps=ks * gparts, nbox=nbox,
                kbb=kbb, Kb=Kb, tok=tok, wbytes=wbytes, pbytes=pbytes, area=area, wblk=wblk, smem=smem)


def test_decode_plan_of_the_decode_workload():
    p = decode_plan(8, 10944, 2048, 152)
    assert (p["R"], p["ctas"], p["groups"], p["ks"], p["gparts"], p["nbox"], p["kbb"], p["tok"]) == \
        (72, 152, 5, 16, 1, 4, 4, 8)
    assert p["smem"] <= DECODE_SMEM_LIMIT
    assert decode_plan(1, 10944, 2048, 152)["ctas"] == 152
    big = decode_plan(16, 38912, 256, 152)   # the widest slices a box holds: 256 rows, 16 row groups
    assert (big["R"], big["groups"], big["ks"], big["gparts"], big["tok"]) == (256, 16, 2, 8, 16)
    assert decode_plan(16, 38912, 256, 148) is None
    # slices too large for shared memory, or more than 16 tokens: the tcgen05 kernels
    for shape in ((8, 24576, 1536), (16, 10944, 7168), (2, 10944, 7168), (17, 576, 7168), (64, 10944, 2048)):
        assert decode_plan(*shape, 152) is None, shape


@pytest.mark.parametrize("M,N,K", [(8, 10944, 2048), (9, 10944, 2048), (16, 33000, 256), (4, 7, 128),
                                   (1, 1217, 640), (7, 3600, 384), (12, 640, 7168), (16, 320, 256),
                                   (5, 2999, 1024), (16, 11000, 384), (2, 32768, 512), (1, 129, 4096)])
@pytest.mark.parametrize("sms", [152, 148, 132])
def test_decode_plan_covers_every_weight_row_and_k_block_once(M, N, K, sms):
    """Every (weight row < N, K block) goes to exactly one warp of one CTA;
    no warp holds more row groups than its accumulators; every box holds at
    least one K block; the staged weight scales cover the slice's 128-row
    blocks; the partials fit in the weight area."""
    p = decode_plan(M, N, K, sms)
    assert p is not None
    R, Kb, G = p["R"], p["Kb"], p["groups"]
    assert R % 8 == 0 and p["ctas"] <= sms and p["warps"] <= 16
    assert (p["nbox"] - 1) * p["kbb"] < Kb <= p["nbox"] * p["kbb"]
    seen = {}
    for c in range(p["ctas"]):
        r0 = c * R
        assert r0 < N
        blocks = min(r0 + R - 1, N - 1) // 128 - r0 // 128 + 1
        assert blocks <= p["wblk"]
        for ks in range(p["ks"]):
            kb0, kb1 = ks * Kb // p["ks"], (ks + 1) * Kb // p["ks"]
            assert kb0 < kb1
            for gp in range(p["gparts"]):
                g0, g1 = gp * G // p["gparts"], (gp + 1) * G // p["gparts"]
                assert 1 <= g1 - g0 <= p["gpw"]
                for r in range(g0 * 16, g1 * 16):
                    if r >= R or r0 + r >= N:
                        continue
                    for kb in range(kb0, kb1):
                        seen[(r0 + r, kb)] = seen.get((r0 + r, kb), 0) + 1
    assert len(seen) == N * Kb and set(seen.values()) == {1}
    assert p["pbytes"] <= p["area"]


def test_decode_plan_mirror_matches_the_library_plan(tmp_path):
    """The mirror above against the plan the library computes: the plan
    function compiled from the kernel's own source (tests/cuda/
    decode_plan_dump.cu, host code only), over a grid of shapes and SM counts
    that includes every refusal (too many tokens, slices past 256 rows or past
    shared memory, K not a multiple of 128)."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    exe = str(tmp_path / "decode_plan_dump")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17",
                    "-I", os.path.join(root, "include"), "-I", os.path.join(root, "fp8_block_scaled_quant_gb300", "csrc"),
                    "-o", exe, os.path.join(here, "cuda", "decode_plan_dump.cu")],
                   check=True, capture_output=True, timeout=300)
    shapes = list(itertools.product((1, 2, 7, 8, 9, 16, 17, 64),
                                    (1, 7, 8, 129, 320, 1217, 2999, 10944, 24576, 32768, 38912, 50000),
                                    (100, 128, 256, 384, 640, 2048, 7168, 12288),
                                    (152, 148, 132, 2, 1)))
    res = subprocess.run([exe], input="\n".join(f"{M} {N} {K} {s}" for M, N, K, s in shapes) + "\n",
                         capture_output=True, text=True, timeout=120)
    lines = res.stdout.splitlines()
    assert res.returncode == 0 and len(lines) == len(shapes)
    taken = 0
    for (M, N, K, sms), line in zip(shapes, lines):
        got = [int(v) for v in line.split()]
        p = decode_plan(M, N, K, sms)
        if p is None:
            assert got[0] == 0, (M, N, K, sms, got)
            continue
        taken += 1
        want = [1, p["R"], p["ctas"], p["groups"], p["ks"], p["gparts"], p["warps"], p["nbox"], p["kbb"], p["wblk"],
                p["smem"]]
        assert got == want, (M, N, K, sms, got, want)
    assert 500 < taken < len(shapes)

