"""The page layout written in include/kvs.h is the layout the library stores.

A caller of kvs_attend_pages_noalloc or kvs_load_host_pages builds pages from
the header alone.  This test reads the byte formulas and sub-array offsets
out of the header's comment text, builds every page of a history with them
(from the oracle's Q8_0 / Q4_0 blocks), and compares with the oracle's page
encoder byte for byte.  The GPU tests pin the library's stored pages to that
same encoder, so the chain header -> encoder -> device bytes is closed.
"""
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_layout():
    text = open(os.path.join(ROOT, "include", "kvs.h")).read()
    i = text.index("Page layout.")
    block = text[i:text.index("*/", i)]
    block = re.sub(r"\n\s*\*\s?", " ", block)  # unwrap the comment lines
    off = dict(re.findall(r"(Kq|Ks|Vq|Vs)\s+offset\s+([0-9P*D/ ]+?),", block))
    kq = re.search(r"int8 Q8_0 code of \(t, d\) at byte\s+(.+?d%32)", block).group(1)
    vq = re.search(r"the byte of \(t, j\) is at\s+(.+?t%32)", block).group(1)
    ks = re.search(r"Q8_0 scale of \(t, block b\)\s+at fp16 element ([tNBb*+ ]+)", block).group(1)
    vs = re.search(r"Q4_0 scale of \(t, block b\)\s+at fp16 element ([tNBbP*+ ]+)", block).group(1)
    lo = re.search(r"packs dims\s+(j/16\*32 \+ j%16) \(low nibble\)", block).group(1)
    sect = re.search(r"Hk head sections of S = ([P*D/0-9]+) bytes", block).group(1)

    def fn(expr, names):
        py = expr.strip().replace("/", "//")
        return eval("lambda " + ", ".join(names) + ": " + py)  # noqa: S307 - header text of this repo

    return dict(kq=fn(kq, "t d NB".split()), vq=fn(vq, "t j NB".split()), ks=fn(ks, "t b NB".split()),
                vs=fn(vs, "t b P".split()), lo=fn(lo, ["j"]), sect=fn(sect, "P D".split()),
                off={k: fn(v, "P D".split()) for k, v in off.items()})


def test_header_states_every_formula():
    lay = _header_layout()
    assert set(lay["off"]) == {"Kq", "Ks", "Vq", "Vs"}
    P, D = 256, 256
    assert lay["sect"](P, D) == P * D * 13 // 8
    assert lay["off"]["Kq"](P, D) == 0


def _page_from_header(lay, qkv, P, Hk, D, T, page):
    NB = D // 32
    S = lay["sect"](P, D)
    out = np.zeros(Hk * S, np.uint8)
    o = {k: f(P, D) for k, f in lay["off"].items()}
    for g in range(Hk):
        base = g * S
        for t in range(P):
            tok = page * P + t
            if tok >= T:
                break
            for d in range(D):
                out[base + o["Kq"] + lay["kq"](t, d, NB)] = np.uint8(qkv.kq[tok, g, d].view(np.uint8))
            for b in range(NB):
                for byte, bits in ((0, qkv.kd[tok, g, b] & 0xFF), (1, qkv.kd[tok, g, b] >> 8)):
                    out[base + o["Ks"] + 2 * lay["ks"](t, b, NB) + byte] = bits
                for byte, bits in ((0, qkv.vd[tok, g, b] & 0xFF), (1, qkv.vd[tok, g, b] >> 8)):
                    out[base + o["Vs"] + 2 * lay["vs"](t, b, P) + byte] = bits
            for j in range(D // 2):
                dl = lay["lo"](j)
                out[base + o["Vq"] + lay["vq"](t, j, NB)] = qkv.vq[tok, g, dl] | (qkv.vq[tok, g, dl + 16] << 4)
    return out


@pytest.mark.parametrize("P,Hk,D,T", [(32, 2, 64, 77), (64, 1, 128, 64 * 2 + 5), (256, 1, 256, 300)])
def test_pages_built_from_the_header_match_the_encoder(P, Hk, D, T):
    lay = _header_layout()
    k = synth.normal(99, synth.tag("K", P), (T, Hk, D))
    v = synth.normal(99, synth.tag("V", P), (T, Hk, D))
    qkv = oracle.QuantKV(k, v)
    for page in range((T + P - 1) // P):
        want = qkv.encode_page(P, page)
        got = _page_from_header(lay, qkv, P, Hk, D, T, page)
        assert np.array_equal(got, want), f"page {page}: {np.flatnonzero(got != want)[:8]}"
