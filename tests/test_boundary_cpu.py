"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def dsa():
    import __graft_entry__
    __graft_entry__.build_library()
    import sparse_attention_score_gb300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_stage_calls():
    syms = declared_symbols()
    for s in ("dsa_index_score", "dsa_topk", "dsa_sparse_attn_decode", "dsa_sparse_attn_prefill"):
        assert s in syms


def test_library_exports_every_declared_symbol(dsa):
    lib = ctypes.CDLL(dsa.LIB_PATH)
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert set(declared_symbols()) == set(dsa.SYMBOLS)


def test_version_and_sizes(dsa):
    assert dsa.version() >= 100
    assert dsa.index_score_workspace_size(32, 64, 128, 32768) >= 256
    assert dsa.topk_workspace_size(32, 32768, 2048) >= 256
    assert dsa.sparse_attn_decode_workspace_size(32, 64, 576, 512, 2048) >= 256
    assert dsa.sparse_attn_prefill_workspace_size(16384, 64, 576, 512, 2048) >= 256


def _layout(dsa, **kw):
    f = dict(block_size=64, num_blocks=16, max_blocks_per_seq=4, batch=2, max_seq_len=200,
             reserved_=0, block_table=0x10000, seq_lens=0x20000)
    f.update(kw)
    return dsa.PagedLayoutC(**{k: v for k, v in f.items()})


FAKE = ctypes.c_void_p(0x100000)   # never dereferenced: every call below fails validation


def test_index_score_rejects_bad_arguments(dsa):
    lib = dsa.lib()
    lay = _layout(dsa)
    ws_ok = dsa.index_score_workspace_size(2, 4, 64, 256)
    args = lambda **o: dict(dict(layout=ctypes.byref(lay), q=FAKE, w=FAKE, k=FAKE, dt=0, H=4, D=64,
                                 qs=None, qp=None, Nq=2, s=FAKE, ld=256, ws=FAKE, wsb=ws_ok,
                                 st=None), **o)

    def call(**o):
        a = args(**o)
        return lib.dsa_index_score(a["layout"], a["q"], a["w"], a["k"], a["dt"], a["H"], a["D"],
                                   a["qs"], a["qp"], a["Nq"], a["s"], a["ld"], a["ws"], a["wsb"],
                                   a["st"])
    assert call(layout=None) == -1
    assert call(q=None) == -1
    assert call(ld=0) == -1
    assert call(Nq=-1) == -1
    assert call(D=48) == -2
    assert call(H=0) == -2
    assert call(dt=7) == -2
    assert call(ws=None) == -3
    assert call(wsb=10) == -3
    assert call(ws=ctypes.c_void_p(0x100010)) == -3
    bad = _layout(dsa, block_size=0)
    assert call(layout=ctypes.byref(bad)) == -1
    bad = _layout(dsa, max_seq_len=4 * 64 + 1)
    assert call(layout=ctypes.byref(bad)) == -1
    assert "max_seq_len" in dsa.lib().dsa_last_error_string().decode()


def test_index_score_bounded_rejects_bad_arguments(dsa):
    """Refused before any launch: NULL tensors, K out of range, unsupported
    shapes, a batch beyond the grid's y dimension, a short workspace."""
    lib = dsa.lib()
    lay = _layout(dsa)
    ok = dsa.index_score_bounded_workspace_size(2, 4, 64, 256, 16)

    def call(layout=None, kb=FAKE, K=16, D=64, ws=FAKE, wsb=ok):
        layout = layout if layout is not None else lay
        return lib.dsa_index_score_bounded(ctypes.byref(layout), FAKE, FAKE, FAKE, 0, 4, D, kb, K,
                                           FAKE, 256, ws, wsb, None)
    assert call(kb=None) == -1
    assert call(K=0) == -1
    assert call(K=70000) == -1
    assert call(D=48) == -2
    big = _layout(dsa, batch=70000)
    assert call(layout=big) == -2
    assert "batch" in lib.dsa_last_error_string().decode()
    assert call(wsb=10) == -3
    assert call(ws=None) == -3


def test_topk_rejects_bad_arguments(dsa):
    lib = dsa.lib()
    ok = dsa.topk_workspace_size(4, 100, 8)
    assert lib.dsa_topk(FAKE, 100, FAKE, 4, 0, FAKE, FAKE, ok, None) == -1
    assert lib.dsa_topk(FAKE, 100, FAKE, 4, 70000, FAKE, FAKE, ok, None) == -1
    assert lib.dsa_topk(None, 100, FAKE, 4, 8, FAKE, FAKE, ok, None) == -1
    assert lib.dsa_topk(FAKE, 0, FAKE, 4, 8, FAKE, FAKE, ok, None) == -1
    assert lib.dsa_topk(FAKE, 100, FAKE, 4, 8, FAKE, None, ok, None) == -3


def test_attention_rejects_bad_arguments(dsa):
    lib = dsa.lib()
    lay = _layout(dsa)
    ok = dsa.sparse_attn_decode_workspace_size(2, 16, 128, 128, 64)

    def dec(Hq=16, Dqk=128, Dv=128, ks=128, vs=128, scale=0.1, q=FAKE, ws=FAKE, wsb=ok):
        return lib.dsa_sparse_attn_decode(ctypes.byref(lay), q, FAKE, ks, FAKE, vs, Hq, Dqk, Dv,
                                          FAKE, 64, scale, FAKE, None, ws, wsb, None)
    assert dec(q=None) == -1
    assert dec(ks=64) == -1
    assert dec(vs=100) == -1
    assert dec(scale=0.0) == -1
    assert dec(scale=float("nan")) == -1
    assert dec(Hq=0) == -2
    assert dec(Dqk=100, ks=104) == -2
    assert dec(wsb=1) == -3
    assert dec(ws=None) == -3
    okp = dsa.sparse_attn_prefill_workspace_size(3, 16, 128, 128, 64)
    assert lib.dsa_sparse_attn_prefill(ctypes.byref(lay), FAKE, FAKE, 128, FAKE, 128, 16, 128,
                                       128, None, None, 3, FAKE, 0, 0.1, FAKE, None, FAKE, okp,
                                       None) == -1


def test_get_status_rejects_null(dsa):
    v = ctypes.c_int32(0)
    assert dsa.lib().dsa_get_status(None, None, ctypes.byref(v), 0) == -1


def test_noalloc_scratch_size_matches_the_header(dsa):
    """The binding's limit for dsa_topk_noalloc is the library's own (queried
    through dsa_topk_noalloc_scratch_bytes), and equals the header's define."""
    m = re.search(r"#define\s+DSA_TOPK_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)",
                  open(HEADER).read())
    assert m, "DSA_TOPK_NOALLOC_SCRATCH_BYTES not found in the header"
    want = int(m.group(1)) << int(m.group(2))
    assert int(dsa.lib().dsa_topk_noalloc_scratch_bytes()) == want
    assert dsa.TOPK_NOALLOC_SCRATCH_BYTES == want


def test_prefill_step_chunked_workspace_holds_one_chunk_of_scores(dsa):
    """dsa_prefill_step_chunked keeps one chunk of scores in its workspace
    instead of the [Nq][ld] score matrix: for a 16384-token prompt the
    automatic chunk is 768 queries (48 MB), against the 1 GiB matrix the staged
    step's caller provides."""
    T, K = 16384, 2048
    staged = dsa.prefill_step_workspace_size(T, 64, 128, T, 64, 576, 512, K)
    auto = dsa.prefill_step_chunked_workspace_size(T, 64, 128, T, 64, 576, 512, K, 0)
    assert auto - staged <= (48 << 20) + (1 << 20)        # plus one chunk of scores
    assert auto - staged >= 768 * T * 4                     # 768 queries of 16384 scores
    assert dsa.prefill_step_chunked_workspace_size(T, 64, 128, T, 64, 576, 512, K, 16) < auto


def test_prefill_step_chunked_rejects_bad_arguments(dsa):
    lib = dsa.lib()
    lay = _layout(dsa)
    ws = ctypes.create_string_buffer(1 << 12)
    base = [ctypes.byref(lay), 0, FAKE, FAKE, 8, FAKE, FAKE, 576, FAKE, FAKE, 576, FAKE, FAKE,
            dsa.DSA_FP8_E4M3, FAKE, FAKE, 64, 128, FAKE, 64, 576, 512, 16, 0.1, 200, 0, FAKE, FAKE,
            FAKE, ctypes.cast(ws, ctypes.c_void_p), len(ws), None]
    def call(over=None):
        a = list(base)
        for k, v in (over or {}).items():
            a[k] = v
        return lib.dsa_prefill_step_chunked(*a)
    before = dsa.launch_count()
    assert call({1: 5}) == -1                     # seq outside the layout
    assert call({25: -1}) == -1                   # chunk < 0
    assert call({13: 99}) == -2                   # unknown indexer dtype
    assert call({26: None}) == -1                 # idx NULL
    assert call() == -3                           # workspace too small
    assert dsa.launch_count() == before           # nothing launched
