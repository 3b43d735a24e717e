"""Host-side checks of the C ABI: the library loads, exports what include/kvq.h declares, prices the
pool correctly, and rejects bad arguments before touching the GPU (no GPU needed)."""
import ctypes
import json
import math
import os
import re

import pytest

import oracle as O
from block_quantized_bit_gb300 import build_lib, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "page_facts.json")))


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return kvq.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(kvq.EXPORTS) == set(names)
    assert kvq.kvq_version() == "0.1.0"


def L(**kw):
    base = dict(num_pages=10, page_size=16, num_kv_heads=2, head_dim=128, v_dim=128, mla=False)
    base.update(kw)
    return kvq.Layout(**base)


@pytest.mark.parametrize("hkv,d,mla", [(8, 128, False), (2, 256, False), (1, 576, True), (4, 64, False)])
def test_cost_model_matches_the_oracle_and_the_pages(lib, hkv, d, mla):
    lay = L(num_kv_heads=hkv, head_dim=d, v_dim=512 if mla else d, mla=mla)
    n_kv = 1 if mla else 2
    bpt = kvq.kvq_bytes_per_token(lay)
    assert bpt == O.bytes_per_token(n_kv, hkv, d)
    assert bpt == GOLDEN["bytes_per_element_8bit"]["value"] * n_kv * hkv * d
    assert kvq.kvq_pool_bytes(lay) == 10 * 16 * n_kv * hkv * d
    assert kvq.kvq_scale_bytes(lay) == 10 * 16 * n_kv * hkv * d // 32 * 2
    budget = 123_456_789
    pages = kvq.kvq_num_pages(lay, budget)
    assert pages == budget // int(16 * bpt)


def test_pool_growth_against_bf16_at_equal_bytes(lib):
    """Pool tokens grow by exactly 32/17 = 2/1.0625 (review comment 'End-to-end numbers': +88%)."""
    lay = L(num_kv_heads=2, head_dim=256, v_dim=256)
    bf16_per_token = 2 * 2 * 2 * 256
    for budget in (10 ** 9, 37 * 10 ** 9, 2 ** 40):
        q_tokens = kvq.kvq_num_pages(lay, budget) * 16
        b_tokens = budget // (bf16_per_token * 16) * 16
        assert abs(q_tokens / b_tokens - 32 / 17) < 1e-4
    pool = GOLDEN["kv_pool_tokens"]
    # a budget of [305730, 305731) bf16 tokens holds [305730, 305731) * 32/17 8-bit tokens
    assert math.floor(pool["bf16"] * 32 / 17) <= pool["fp8_e4m3"] <= math.floor((pool["bf16"] + 1) * 32 / 17)


def test_invalid_layouts_are_rejected(lib):
    assert kvq.kvq_pool_bytes(L(head_dim=100, v_dim=100)) == 0
    assert kvq.kvq_bytes_per_token(L(head_dim=0, v_dim=0)) == -1.0
    assert kvq.kvq_num_pages(L(num_kv_heads=0), 10 ** 6) == -1
    assert kvq.kvq_decode_workspace_bytes(L(), 4, 7, 10) == 0       # Hq % Hkv != 0
    assert kvq.kvq_decode_workspace_bytes(L(), 4, 8, 10) > 0


FAKE = 0x10000  # an aligned host address that must never be dereferenced: validation fails first


def _store(lib, layout, kind=1, k=FAKE, v=FAKE, sm=FAKE, pool=FAKE, scales=FAKE, n=4):
    P = ctypes.c_void_p
    return lib.kvq_store(P(pool), P(scales), P(k), P(v) if v else None, P(sm), n, ctypes.byref(layout.c()), kind,
                         None)


def test_store_argument_errors(lib):
    assert _store(lib, L(), kind=3) == -2                        # KVQ_EKIND
    assert _store(lib, L(head_dim=48, v_dim=48)) == -3           # KVQ_EHEADDIM
    assert _store(lib, L(), k=0) == -1                           # null k
    assert _store(lib, L(), v=0) == -1                           # GQA needs v
    assert _store(lib, L(mla=True, num_kv_heads=1, head_dim=576, v_dim=512)) == -1   # MLA must not pass v
    assert _store(lib, L(), k=FAKE + 8) == -4                    # KVQ_EALIGN
    assert _store(lib, L(), pool=FAKE + 4) == -4
    assert _store(lib, L(), n=-1) == -1
    assert _store(lib, L(), n=0) == 0                            # nothing to do, nothing launched


def _decode(lib, layout, *, q=FAKE, ws_bytes=None, batch=2, hq=8, maxp=10, kind=1, out_dtype=0, ws=FAKE, opts=None):
    P = ctypes.c_void_p
    if ws_bytes is None:
        ws_bytes = lib.kvq_decode_workspace_bytes(ctypes.byref(layout.c()), batch, hq, maxp)
    o = ctypes.byref(opts) if opts is not None else None
    return lib.kvq_decode_ex(P(q), P(FAKE), P(FAKE), P(FAKE), maxp, P(FAKE), batch, hq, 1.0, P(FAKE), out_dtype,
                             P(ws), ws_bytes, ctypes.byref(layout.c()), kind, o, None)


def test_decode_argument_errors(lib):
    assert _decode(lib, L(), kind=0) == -2
    assert _decode(lib, L(), hq=7) == -1
    assert _decode(lib, L(), ws_bytes=16) == -5                  # KVQ_EWORKSPACE
    assert _decode(lib, L(), q=FAKE + 2) == -4                   # KVQ_EALIGN
    assert _decode(lib, L(), ws=FAKE + 8) == -4
    assert _decode(lib, L(), out_dtype=5) == -1
    assert _decode(lib, L(page_size=32)) == -8                   # KVQ_EUNSUPPORTED
    assert _decode(lib, L(head_dim=96, v_dim=96)) == -8
    assert _decode(lib, L(), batch=0) == 0
    bad = kvq.kvq_decode_options(-3, 0)
    assert _decode(lib, L(), opts=bad) == -1


def _extend(lib, layout, *, hq=8, kind=1, sm_scale=1.0, ws=FAKE, ws_bytes=256, total_q=5, batch=2, out_dtype=0,
            path=None):
    P = ctypes.c_void_p
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), 10, P(FAKE), P(FAKE), total_q, batch, hq, ctypes.c_float(sm_scale),
            P(FAKE), out_dtype, P(ws), ws_bytes, ctypes.byref(layout.c()), kind)
    if path is None:
        return lib.kvq_extend(*args, None)
    return lib.kvq_extend_ex(*args, ctypes.byref(kvq.kvq_extend_options(path)), None)


def _extend_ws(lib, layout, total_q, hq, max_pages, path=None):
    opts = None if path is None else ctypes.byref(kvq.kvq_extend_options(path))
    return lib.kvq_extend_workspace_bytes_ex(ctypes.byref(layout.c()), total_q, hq, max_pages, opts)


def test_extend_kernel_choice(lib):
    """The flash kernel where it supports the shape, else the prefixes on the decode's own choice; path 1
    forces the CUDA-core decode (fp32 P), path 2 the flash kernel (GQA) or the tensor-core decode (MLA)."""
    def path(layout, total_q=5, hq=8, max_pages=10, opt=None, precise=0):
        o = None if opt is None and not precise else ctypes.byref(kvq.kvq_extend_options(opt or 0, precise))
        return lib.kvq_extend_path(ctypes.byref(layout.c()), total_q, hq, max_pages, o)
    assert path(L()) == 3
    assert path(L(), opt=1) == 1
    assert path(L(), opt=2) == 3
    assert path(L(head_dim=64, v_dim=64)) == 1                  # no flash kernel: the decode's choice
    assert path(L(head_dim=64, v_dim=64), opt=2) == -8
    assert path(L(), hq=6) == 1                                 # 3 heads per kv head: CUDA-core decode
    assert path(L(num_kv_heads=2), hq=24) == 2                  # 12 heads per kv head: tensor-core decode
    assert path(L(num_kv_heads=2), hq=24, opt=1) == 1
    mla = L(mla=True, num_kv_heads=1, head_dim=576, v_dim=512)
    assert path(mla, hq=16) == 1                                # 5 prefixes x 160 tokens: below the MLA cutoff
    assert path(mla, total_q=2048, hq=16) == 2                  # chunks of 1024 prefixes
    assert path(mla, total_q=2048, hq=16, opt=1) == 1
    assert path(mla, hq=16, opt=2) == 2
    assert path(L(), opt=5) == -1
    assert path(L(page_size=32)) == -8
    # precise_p: the flash kernel with P as two bf16 terms; prefixes only on the CUDA-core decode
    assert path(L(), precise=1) == 4
    assert path(L(), opt=2, precise=1) == 4
    assert path(L(), opt=1, precise=1) == 1
    assert path(L(head_dim=64, v_dim=64), precise=1) == 1
    assert path(L(num_kv_heads=2), hq=24, precise=1) == 1
    assert path(mla, total_q=2048, hq=16, precise=1) == 1
    assert path(mla, hq=16, opt=2, precise=1) == -8
    assert _extend_ws(lib, L(), 5, 8, 10) == lib.kvq_extend_workspace_bytes_ex(
        ctypes.byref(L().c()), 5, 8, 10, ctypes.byref(kvq.kvq_extend_options(0, 1)))


def test_extend_argument_errors(lib):
    """Everything the host can check is checked before the status word is cleared (no device needed)."""
    assert lib.kvq_extend_workspace_bytes() == 256
    assert _extend(lib, L(), kind=0) == -2                      # KVQ_EKIND
    assert _extend(lib, L(), hq=7) == -1                        # not a multiple of the kv heads
    assert _extend(lib, L(), sm_scale=0.0) == -1                # the softmax scale must be > 0
    assert _extend(lib, L(), sm_scale=-0.5) == -1
    assert _extend(lib, L(), sm_scale=float("nan")) == -1
    assert _extend(lib, L(), total_q=-1) == -1
    assert _extend(lib, L(), out_dtype=7) == -1
    # head_dim 64 and 3 heads per kv head have no flash kernel: the prefixes take them, with their workspace
    assert _extend(lib, L(head_dim=64, v_dim=64)) == -5
    assert _extend(lib, L(), hq=6) == -5
    assert _extend(lib, L(), hq=6, path=2) == -8                # the flash kernel asked for: KVQ_EUNSUPPORTED
    assert _extend(lib, L(), path=3) == -1
    assert _extend(lib, L(head_dim=96, v_dim=96), ws_bytes=1 << 30) == -8
    mla = L(mla=True, num_kv_heads=1, head_dim=576, v_dim=512)
    need = _extend_ws(lib, mla, 5, 16, 10)
    assert need > 256                                           # the decode workspace of the prefixes
    assert _extend_ws(lib, L(), 5, 8, 10) == 256
    assert _extend_ws(lib, L(), 5, 8, 10, path=1) > 256
    assert _extend_ws(lib, mla, -1, 16, 10) == 0
    assert _extend_ws(lib, L(), 5, 8, 10, path=-1) == 0
    assert _extend(lib, mla, hq=16) == -5                       # MLA with the flash kernel's workspace: too small
    assert _extend(lib, mla, hq=16, ws_bytes=need, ws=FAKE + 8) == -4
    assert _extend(lib, L(mla=True, num_kv_heads=1, head_dim=512, v_dim=512), hq=16, ws_bytes=1 << 30) == -8
    assert _extend(lib, L(page_size=32)) == -8
    assert _extend(lib, L(), ws_bytes=16) == -5                 # KVQ_EWORKSPACE
    assert _extend(lib, L(), ws=FAKE + 8) == -4                 # KVQ_EALIGN


def _sparse(lib, layout, *, topk=256, hq=8, kind=1, out_dtype=0, ws=FAKE, ws_bytes=None, ix=FAKE, batch=2):
    P = ctypes.c_void_p
    if ws_bytes is None:
        ws_bytes = lib.kvq_decode_sparse_workspace_bytes(ctypes.byref(layout.c()), batch, hq, topk)
    return lib.kvq_decode_sparse(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 10, P(FAKE), P(ix), topk, batch, hq,
                                 ctypes.c_float(1.0), P(FAKE), out_dtype, P(ws), ws_bytes, ctypes.byref(layout.c()),
                                 kind, None)


def test_sparse_decode_argument_errors(lib):
    """Checked on the host before any device call (no GPU needed)."""
    lay = L()
    assert lib.kvq_decode_sparse_workspace_bytes(ctypes.byref(lay.c()), 2, 8, 256) > 0
    assert lib.kvq_decode_sparse_workspace_bytes(ctypes.byref(lay.c()), 2, 8, 8193) == 0   # above the 8192 cap
    assert lib.kvq_decode_sparse_workspace_bytes(ctypes.byref(lay.c()), 2, 8, -1) == 0
    assert _sparse(lib, lay, kind=9) == -2                      # KVQ_EKIND
    assert _sparse(lib, lay, out_dtype=4) == -1
    assert _sparse(lib, lay, topk=8193, ws_bytes=1 << 30) == -1
    assert _sparse(lib, lay, hq=7, ws_bytes=1 << 30) == -1      # not a multiple of the kv heads
    assert _sparse(lib, L(head_dim=96, v_dim=96), ws_bytes=1 << 30) == -8   # head_dim not a multiple of 64
    assert _sparse(lib, lay, ws_bytes=64) == -5                 # KVQ_EWORKSPACE
    assert _sparse(lib, lay, ws=FAKE + 8) == -4                 # KVQ_EALIGN
    assert _sparse(lib, lay, ix=FAKE + 2) == -4
    assert _sparse(lib, lay, batch=0) == 0


def test_wait_probe_argument_errors(lib):
    assert lib.kvq_wait_probe(None, None) == -1                 # no workspace
    assert lib.kvq_wait_probe(ctypes.c_void_p(FAKE + 4), None) == -4


def test_workspace_bound_covers_every_split_choice(lib):
    lay = L(num_kv_heads=8, head_dim=128, v_dim=128)
    auto = kvq.kvq_decode_workspace_bytes(lay, 8, 16, 1024)
    forced = kvq.kvq_decode_workspace_bytes(lay, 8, 16, 1024, pages_per_split=1)
    assert forced > auto > 0


def test_decode_path_follows_the_group_size_and_the_options(lib):
    mla = L(num_kv_heads=1, head_dim=576, v_dim=512, mla=True)
    assert kvq.kvq_decode_path(L(num_kv_heads=8), 8, 16, 1024) == 1                          # G = 2: CUDA cores
    assert kvq.kvq_decode_path(L(num_kv_heads=2, head_dim=256, v_dim=256), 8, 16, 64) == 2  # G = 8: tcgen05
    assert kvq.kvq_decode_path(mla, 1, 128, 10240) == 2                                     # long MLA context
    assert kvq.kvq_decode_path(mla, 1, 128, 16) == 1                                        # 256 tokens at most
    assert kvq.kvq_decode_path(mla, 4, 128, 16) == 2                                        # 4 x 256 tokens
    assert kvq.kvq_decode_path(mla, 1, 128, 16, path=2) == 2                                # forced
    assert kvq.kvq_decode_path(L(num_kv_heads=2, head_dim=256, v_dim=256), 8, 16, 64, path=1) == 1
    assert kvq.kvq_decode_path(L(num_kv_heads=8, head_dim=64, v_dim=64), 8, 16, 64, path=2) == -8  # unsupported
    assert kvq.kvq_decode_path(L(), 4, 7, 64) == -1                                         # Hq % Hkv != 0
    assert kvq.kvq_decode_path(L(), 4, 8, 64, path=3) == -1
    assert kvq.kvq_decode_path(L(), 4, 8, 0) == -1


def test_strerror_has_a_message_for_every_status(lib):
    for code, name in kvq.STATUS.items():
        msg = kvq.strerror(code)
        assert msg and msg != "unknown status", name


def test_the_product_path_has_no_fallback(monkeypatch):
    """Without the built library every call raises: there is no CPU path to fall back on.  And the product
    package never imports the oracle."""
    monkeypatch.setattr(kvq, "LIB_PATH", os.path.join(os.path.dirname(build_lib.LIB), "missing", "libkvq.so"))
    monkeypatch.setattr(kvq, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        kvq.lib()
    with pytest.raises(RuntimeError, match="not built"):
        kvq.alloc_extend_workspace("cpu")
    pkg = os.path.dirname(kvq.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "kvq_oracle" not in text, f


def test_fused_store_argument_errors(lib):
    P = ctypes.c_void_p
    mla = L(num_kv_heads=1, head_dim=576, v_dim=512, mla=True)

    def call(layout=mla, kind=1, rope=64, kv=FAKE, n=4):
        return lib.kvq_store_act_quant(P(FAKE), P(FAKE), P(kv), P(FAKE), n, rope, ctypes.byref(layout.c()), kind, None)

    assert call(kind=5) == -2                                   # KVQ_EKIND
    assert call(layout=L()) == -1                               # a GQA pool: not this store
    assert call(rope=32) == -8                                  # rope_dim not a multiple of 64
    assert call(layout=L(num_kv_heads=1, head_dim=544, v_dim=512, mla=True)) == -8
    assert call(n=-1) == -1
    assert call(n=0) == 0
    assert call(kv=FAKE + 8) == -4                              # KVQ_EALIGN


def test_unscaled_store_argument_errors(lib):
    P = ctypes.c_void_p

    def call(layout=None, kind=3, v=FAKE, n=4, k=FAKE):
        layout = layout or L()
        return lib.kvq_store_unscaled(P(FAKE), P(k), P(v) if v else None, P(FAKE), n, ctypes.byref(layout.c()), kind,
                                      None)

    assert call(kind=1) == -2                                   # the block-scaled kinds use kvq_store
    assert call(kind=5) == -2
    assert call(layout=L(head_dim=48, v_dim=48)) == -3          # KVQ_EHEADDIM
    assert call(v=0) == -1                                      # GQA needs v
    assert call(layout=L(mla=True, num_kv_heads=1, head_dim=576, v_dim=512)) == -1  # MLA must not pass v
    assert call(n=-1) == -1
    assert call(n=0) == 0
    assert call(k=FAKE + 4) == -4                               # KVQ_EALIGN
    assert call(kind=4) != -2                                   # e5m2 is accepted (fails later: no device here)
    # the decode reads unscaled pools without a scale array (NULL scales pass validation; no device here)
    for kind in (3, 4):
        st = lib.kvq_decode(P(FAKE), P(FAKE), None, P(FAKE), 10, P(FAKE), 2, 8, ctypes.c_float(1.0), P(FAKE), 0,
                            P(FAKE), 1 << 20, ctypes.byref(L().c()), kind, None)
        assert st not in (-1, -2), st
    # the block-scaled kinds still need their scales; an unknown kind is rejected
    assert lib.kvq_decode(P(FAKE), P(FAKE), None, P(FAKE), 10, P(FAKE), 2, 8, ctypes.c_float(1.0), P(FAKE), 0,
                          P(FAKE), 1 << 20, ctypes.byref(L().c()), 1, None) == -1
    assert lib.kvq_decode(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 10, P(FAKE), 2, 8, ctypes.c_float(1.0), P(FAKE), 0,
                          P(FAKE), 1 << 20, ctypes.byref(L().c()), 5, None) == -2


def test_unscaled_cost_model_is_one_byte_per_element_and_doubles_the_bf16_budget(lib):
    """"Add fp8 KV-cache quantization (--kv-dtype)", section "Benchmark": at the same budget the unscaled fp8 pool
    holds twice the bf16 tokens (27,142 -> 54,284); the block-scaled kinds keep 17/16 bytes per element."""
    g = GOLDEN["unscaled_fp8_kv_budget_tokens"]
    for hkv, d in ((8, 128), (2, 256), (4, 64)):
        lay = L(num_kv_heads=hkv, head_dim=d, v_dim=d)
        for kind in ("fp8_e4m3_unscaled", "fp8_e5m2_unscaled"):
            assert kvq.kvq_bytes_per_token_ex(lay, kind) == 2 * hkv * d * O.bytes_per_element(kind)
            bf16_per_page = 16 * 2 * hkv * d * GOLDEN["bytes_per_element_bf16"]["value"]
            budget = g["bf16"] * bf16_per_page // 16        # a budget of exactly 27,142 bf16 tokens (whole pages)
            assert kvq.kvq_num_pages_ex(lay, kind, budget) * 16 == 2 * (budget // bf16_per_page) * 16
        for kind in ("fp8_e4m3", "q8_0"):
            assert kvq.kvq_bytes_per_token_ex(lay, kind) == kvq.kvq_bytes_per_token(lay)
            assert kvq.kvq_num_pages_ex(lay, kind, 10 ** 9) == kvq.kvq_num_pages(lay, 10 ** 9)
        assert kvq.kvq_bytes_per_token_ex(lay, 7) == -1.0 and kvq.kvq_num_pages_ex(lay, 0, 10 ** 9) == -1
    assert g["fp8_e4m3"] == 2 * g["bf16"]


def test_exp2_probe_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.kvq_exp2_probe(P(FAKE), P(FAKE), -1, None) == -1
    assert lib.kvq_exp2_probe(None, P(FAKE), 4, None) == -1
    assert lib.kvq_exp2_probe(P(FAKE), P(FAKE), 0, None) == 0
    assert lib.kvq_exp2_probe(P(FAKE + 2), P(FAKE), 4, None) == -4
