"""Pins for the PRP oracle: worked cases, brute force, invariants, scan.

Follows the xNVMe "uPCIe CUDA" backend page (introduction: 64 KiB LUT,
4 KiB PRP entries; "Limitations": 512-entry list page, 513 x 4 KiB).
"""

import numpy as np
import pytest

from conftest import h, load_golden

PAGE = 4096


def golden_lut(fx):
    n = fx["heap_size"] // 65536
    lut = [0x900000000 + c * 0x30000 for c in range(n)]
    for c, v in enumerate(fx["lut_explicit"]):
        lut[c] = h(v)
    return np.array(lut, dtype=np.uint64)


def golden_cases():
    fx = load_golden("prp_hand_cases.json")
    return [(fx, c) for c in fx["cases"]]


@pytest.mark.parametrize("fx,case", golden_cases(), ids=lambda v: v.get("name", "") if isinstance(v, dict) and "name" in v else "")
def test_hand_cases(oracle, fx, case):
    lut = golden_lut(fx)
    cap = case.get("arena_cap_pages", fx["arena_cap_pages"])
    req = np.array([[h(o), int(n)] for o, n in case["req"]], dtype=np.uint64)
    FILL = 0xDEADBEEFDEADBEEF
    out = oracle.prp_build(req, lut, fx["heap_size"], h(fx["arena_base"]), cap, fill=FILL)
    want = np.array([[h(a), h(b)] for a, b in case["prp"]], dtype=np.uint64)
    assert (out["prp"] == want).all(), [list(map(hex, r)) for r in out["prp"]]
    assert out["page_base"].tolist() == case["page_base"]
    assert out["status"].tolist() == case["status"]
    assert int(out["ctr"][0]) == case["total_pages"]
    assert int(out["ctr"][1]) == case["status"].count(1)
    assert int(out["ctr"][2]) == case["status"].count(2)
    for lp in case["lists"]:
        for slot, val in lp["slots"].items():
            got = int(out["arena"][lp["page"], int(slot)])
            assert got == h(val), (lp["page"], slot, hex(got), val)
    if not case["lists"]:
        assert (out["arena"] == FILL).all()


def brute_force_pages(off, length, lut):
    """Walk every byte of [off, off+len), map it through the LUT, and list the
    distinct 4 KiB bus pages in the order the bytes reach them."""
    b = np.arange(off, off + length, dtype=np.uint64)
    bus = lut[(b >> np.uint64(16)).astype(np.int64)] + (b & np.uint64(0xFFFF))
    pages = bus & ~np.uint64(PAGE - 1)
    change = np.ones(pages.shape[0], dtype=bool)
    change[1:] = pages[1:] != pages[:-1]
    return pages[change]


def data_entries(prp1, prp2, lst, n_list, arena_base, page_base, fill=0):
    """The page entries a request describes, chain pointers removed. On the
    last list page the entries end at the first slot still holding ``fill``
    (never written)."""
    if n_list == 0:
        return [prp1] + ([prp2] if prp2 else [])
    out = [prp1]
    for j in range(n_list):
        for s in range(512):
            v = int(lst[j, s])
            if s == 511 and j + 1 < n_list:
                assert v == arena_base + (page_base + j + 1) * PAGE
                continue
            if j + 1 == n_list and v == fill:
                break
            out.append(v)
    return out


def random_lut(rng, n):
    frames = rng.choice(np.arange(1, 1 << 20, dtype=np.uint64), size=n, replace=False)
    return frames << np.uint64(16)


def test_brute_force_tiny_heaps(oracle):
    rng = np.random.default_rng(1234)
    heap = 4 * 1024 * 1024
    lut = random_lut(rng, heap // 65536)
    A = 0x40000000000
    for trial in range(300):
        off = 4 * int(rng.integers(0, heap // 4))
        length = int(rng.integers(1, min(heap - off, 3 * 1024 * 1024) + 1))
        pb = int(rng.integers(0, 1000))
        prp1, prp2, lst = oracle.prp_one(off, length, lut, heap, A, pb, fill=0xAAAAAAAAAAAAAAAA)
        n_list = lst.shape[0]
        got = data_entries(prp1, prp2, lst, n_list, A, pb, fill=0xAAAAAAAAAAAAAAAA)
        pages = brute_force_pages(off, length, lut)
        # PRP1 keeps its in-page offset; it names the first page.
        assert got[0] & ~(PAGE - 1) == int(pages[0])
        assert got[0] % PAGE == off % PAGE
        # All later entries are exactly the later pages, in order.
        assert [int(x) for x in got[1:]] == [int(x) for x in pages[1:]], (off, length)
        n = len(pages)
        if n >= 3:
            assert prp2 == A + pb * PAGE
        # Unused slots of the last list page stay untouched.
        if n_list:
            used = (n - 1) - 511 * (n_list - 1)
            assert 1 <= used <= 512
            assert (lst[-1, used:] == 0xAAAAAAAAAAAAAAAA).all()


def test_page_count_boundaries(oracle):
    heap = 16 * 1024 * 1024
    # list pages as a function of the page count n (list entries m = n - 1)
    for n, want in [(1, 0), (2, 0), (3, 1), (513, 1), (514, 2), (1023, 2), (1024, 2),
                    (1025, 3), (1534, 3), (1535, 3), (1536, 4)]:
        assert oracle.prp_list_pages(0, n * PAGE, heap) == want, n
    # an unaligned start adds a page
    assert oracle.prp_list_pages(4, 2 * PAGE, heap) == 1
    assert oracle.prp_list_pages(4, 2 * PAGE - 4, heap) == 0
    # the largest 32-bit length
    assert oracle.prp_list_pages(0, 0xFFFFFFFF, 1 << 33) == -(-((1 << 20) - 1) // 511)


def test_invariants_random_batch(oracle):
    """Alignment, span = length, consecutive heap pages, chain pointers, scan."""
    rng = np.random.default_rng(99)
    heap = 64 * 1024 * 1024
    lut = random_lut(rng, heap // 65536)
    inverse = {int(v): c for c, v in enumerate(lut)}
    A = 0x1_0000_0000
    n = 400
    off = 4 * rng.integers(0, heap // 4, size=n).astype(np.uint64)
    length = rng.integers(1, 3 * 1024 * 1024, size=n).astype(np.uint64)
    length = np.minimum(length, np.uint64(heap) - off)
    length[::37] = 0          # a few invalid ones
    req = np.stack([off, length], axis=1).astype(np.uint64)
    out = oracle.prp_build(req, lut, heap, A, 10_000)
    pages = [oracle.prp_list_pages(int(o), int(l), heap) for o, l in req]
    # Textbook: page bases are the exclusive prefix sum of list pages.
    assert out["page_base"].tolist() == (np.cumsum(pages) - pages).tolist()
    assert int(out["ctr"][0]) == sum(pages)
    for i in range(n):
        o, l = int(off[i]), int(length[i])
        if l == 0:
            assert out["status"][i] == 1 and (out["prp"][i] == 0).all()
            continue
        pb = int(out["page_base"][i])
        ents = data_entries(int(out["prp"][i, 0]), int(out["prp"][i, 1]),
                            out["arena"][pb:pb + pages[i]], pages[i], A, pb)
        # every entry after PRP1 is 4 KiB aligned
        assert all(e % PAGE == 0 for e in ents[1:])
        # the span of all entries equals the request length
        span = min(PAGE - o % PAGE, l)
        for k in range(1, len(ents)):
            span += min(PAGE, o + l - (o - o % PAGE + k * PAGE))
        assert span == l
        # entries map back to consecutive heap pages
        heap_pages = [(inverse[e & ~0xFFFF] << 4) | ((e & 0xFFFF) >> 12) for e in ents]
        assert heap_pages == list(range(heap_pages[0], heap_pages[0] + len(ents)))
        assert heap_pages[0] == o // PAGE


def test_zero_tail(oracle):
    rng = np.random.default_rng(5)
    heap = 8 * 1024 * 1024
    lut = random_lut(rng, heap // 65536)
    req = np.array([[0, 20 * PAGE], [4, 600 * PAGE]], dtype=np.uint64)
    out = oracle.prp_build(req, lut, heap, 0x1000000, 8, zero_tail=True, fill=7)
    # request 0: 19 entries on page 0, zeros after
    assert (out["arena"][0, 19:] == 0).all() and (out["arena"][0, :19] != 0).all()
    # request 1: n = 601, 600 entries -> 511 + ptr, then 89 entries + zeros
    assert (out["arena"][2, 89:] == 0).all() and (out["arena"][2, :89] != 0).all()
    assert (out["arena"][3:] == 7).all()


def test_unused_slots_untouched(oracle):
    """Without DB_PRP_ZERO_TAIL every slot after a list's last entry keeps
    what the arena held, whatever the entry count modulo a store width."""
    rng = np.random.default_rng(6)
    heap = 8 * 1024 * 1024
    lut = random_lut(rng, heap // 65536)
    FILL = 7
    req = np.array([[0, 20 * PAGE], [0, 21 * PAGE], [4, 600 * PAGE], [0, 5 * PAGE]],
                   dtype=np.uint64)
    out = oracle.prp_build(req, lut, heap, 0x1000000, 8, fill=FILL)
    a = out["arena"]
    # 19 entries
    assert (a[0, :19] != FILL).all() and (a[0, 19:] == FILL).all()
    # 20 entries
    assert (a[1, :20] != FILL).all() and (a[1, 20:] == FILL).all()
    # 600 entries: 511 + pointer, then 89 entries
    assert (a[2] != FILL).all()
    assert (a[3, :89] != FILL).all() and (a[3, 89:] == FILL).all()
    # 4 entries
    assert (a[4, :4] != FILL).all() and (a[4, 4:] == FILL).all()
    assert (a[5:] == FILL).all()


def test_empty_batch(oracle):
    lut = np.array([0x10000], dtype=np.uint64)
    out = oracle.prp_build(np.zeros((0, 2), dtype=np.uint64), lut, 65536, 0, 4)
    assert out["ctr"].tolist() == [0, 0, 0, 0]
