"""The C-ABI library: loads, exports what include/mla.h declares, validates
arguments on the host.  No kernel is launched here (runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def mla():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_mla_build", os.path.join(ROOT, "head_latent_attention_27_b300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import head_latent_attention_27_b300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mla_cache_append", "mla_decode", "mla_decode_split_combine",
                     "mla_decode_workspace_size", "mla_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(mla):
    lib = ctypes.CDLL(mla.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(mla.EXPORTED)


def test_status_strings(mla):
    for code in range(6):
        assert mla.mla_status_string(code).startswith("MLA_")
    assert "unknown" in mla.mla_status_string(99)


def test_workspace_size_is_host_arithmetic(mla):
    n0 = mla.mla_decode_workspace_size(64, 1, 128, 512, 0, 148)
    n32 = mla.mla_decode_workspace_size(4, 1, 128, 512, 32, 148)
    # balanced: at most units + workers pieces of 128 x 512 fp32 partial rows
    assert n0 >= (64 + 148) * 128 * 512 * 4
    assert n32 >= 4 * 32 * 128 * 512 * 4
    assert mla.mla_decode_workspace_size(64, 2, 128, 512, 0, 148) > n0
    with pytest.raises(RuntimeError):
        mla.mla_decode_workspace_size(0, 0, 128, 512, 0, 148)
    with pytest.raises(RuntimeError):
        mla.mla_decode_workspace_size(4, 1, 128, 512, 5000, 148)


def _cache(mla, **kw):
    c = dict(data=0x1000, page_table=0x2000, dtype=mla.MLA_BF16, num_seqs=4, num_pages=16, page_size=64,
             d_c=512, d_r=64, max_pages_per_seq=4)
    c.update(kw)
    return mla.mla_cache_t(**c)


def _decode(mla, cache, B=2, Q=1, H=128, ws_bytes=1 << 30, seq=0x3000, qn=0x4000, qr=0x5000, out=0x6000,
            ws=0x100000):
    return mla._lib.mla_decode(ctypes.byref(cache), seq, B, qn, qr, Q, H, 0.07, out, None, ws, ws_bytes, None)


def test_decode_rejects_bad_arguments_before_launch(mla):
    E = mla
    assert mla._lib.mla_decode(None, 0x3000, 2, 0x4000, 0x5000, 1, 128, 0.07, 0x6000, None, 0x100000, 1 << 30,
                               None) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla, data=None)) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla, page_size=32)) == E.MLA_ERR_UNSUPPORTED
    assert _decode(mla, _cache(mla, d_c=256)) == E.MLA_ERR_UNSUPPORTED
    assert _decode(mla, _cache(mla, d_r=63)) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla, dtype=7)) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla, data=0x1008)) == E.MLA_ERR_INVALID_ARG     # not 16-byte aligned
    assert _decode(mla, _cache(mla), B=5) == E.MLA_ERR_INVALID_ARG              # B > num_seqs
    assert _decode(mla, _cache(mla), Q=0) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla), H=0) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla), Q=64, H=128) == E.MLA_ERR_UNSUPPORTED      # Q*H > 4096
    assert _decode(mla, _cache(mla), qn=None) == E.MLA_ERR_INVALID_ARG
    assert _decode(mla, _cache(mla), out=0x6004) == E.MLA_ERR_INVALID_ARG      # misaligned out
    assert _decode(mla, _cache(mla, dtype=mla.MLA_FP32, d_c=66, d_r=16)) == E.MLA_ERR_UNSUPPORTED
    assert _decode(mla, _cache(mla, num_pages=0)) == E.MLA_ERR_INVALID_ARG
    c = _cache(mla)
    assert mla._lib.mla_decode_split_combine(ctypes.byref(c), 0x3000, 2, 0x4000, 0x5000, 1, 128, 0.07, 0,
                                             0x6000, None, 0x100000, 1 << 30, None) == E.MLA_ERR_INVALID_ARG
    assert mla._lib.mla_decode_split_combine(ctypes.byref(c), 0x3000, 2, 0x4000, 0x5000, 1, 128, 0.07, 2000,
                                             0x6000, None, 0x100000, 1 << 30, None) == E.MLA_ERR_INVALID_ARG


def test_append_rejects_bad_arguments_before_launch(mla):
    c = _cache(mla)
    f = mla._lib.mla_cache_append
    ok_args = dict(ckv=0x7000, kr=0x8000, dt=mla.MLA_BF16, seq=0x9000, pos=0xA000, T=4, flags=3)

    def call(**kw):
        a = dict(ok_args)
        a.update(kw)
        return f(ctypes.byref(c), a["ckv"], a["kr"], a["dt"], None, 1e-6, 10000.0, a["seq"], a["pos"], a["T"],
                 a["flags"], None)

    assert call(T=-1) == mla.MLA_ERR_INVALID_ARG
    assert call(T=0) == mla.MLA_OK                    # no-op, launches nothing
    assert call(ckv=None) == mla.MLA_ERR_INVALID_ARG
    assert call(seq=None) == mla.MLA_ERR_INVALID_ARG
    assert call(dt=5) == mla.MLA_ERR_INVALID_ARG
    assert call(flags=8) == mla.MLA_ERR_INVALID_ARG
    assert f(None, 0x7000, 0x8000, 0, None, 1e-6, 1e4, 0x9000, 0xA000, 4, 3, None) == mla.MLA_ERR_INVALID_ARG


def test_zero_batch_decode_is_a_no_op(mla):
    c = _cache(mla)
    assert _decode(mla, c, B=0, seq=None, qn=None, qr=None, out=None) == mla.MLA_OK


def test_append_rope_rejects_bad_rope_parameters_before_launch(mla):
    c = _cache(mla)
    f = mla._lib.mla_cache_append_rope

    def call(rope, flags=3, T=4):
        return f(ctypes.byref(c), 0x7000, 0x8000, mla.MLA_BF16, None, 1e-6, ctypes.byref(rope) if rope else None,
                 0x9000, 0xA000, T, flags, None)

    assert call(mla.yarn_rope(base=0.0)) == mla.MLA_ERR_INVALID_ARG
    assert call(mla.yarn_rope(factor=0.5)) == mla.MLA_ERR_INVALID_ARG
    assert call(mla.yarn_rope(alpha=32.0, beta=32.0)) == mla.MLA_ERR_INVALID_ARG
    assert call(mla.yarn_rope(original_max_position=0)) == mla.MLA_ERR_INVALID_ARG
    assert call(None) == mla.MLA_ERR_INVALID_ARG                    # RoPE requested without parameters
    assert call(mla.yarn_rope(), T=0) == mla.MLA_OK                # no-op, launches nothing
    assert call(mla.yarn_rope(), T=-1) == mla.MLA_ERR_INVALID_ARG


def test_yarn_softmax_scale_is_host_arithmetic(mla):
    assert abs(mla.mla_yarn_softmax_scale(1.0, 40.0) - (0.0707 * __import__("math").log(40.0) + 1.0) ** 2) < 1e-6
    assert mla.mla_yarn_softmax_scale(0.25, 1.0) == 0.25


def test_absorb_rejects_bad_arguments_before_launch(mla):
    for fn in (mla._lib.mla_absorb_query, mla._lib.mla_absorb_output):
        def call(w=0x10000, x=0x20000, y=0x30000, n=64, H=128, d_h=128, d_c=512):
            return fn(w, x, y, n, H, d_h, d_c, None, None)

        assert call(n=0, w=None, x=None, y=None) == mla.MLA_OK      # empty: no launch
        assert call(n=-1) == mla.MLA_ERR_INVALID_ARG
        assert call(H=0) == mla.MLA_ERR_INVALID_ARG
        assert call(d_h=64) == mla.MLA_ERR_UNSUPPORTED               # d_h, d_c multiples of 128
        assert call(d_c=320) == mla.MLA_ERR_UNSUPPORTED
        assert call(w=None) == mla.MLA_ERR_INVALID_ARG
        assert call(x=None) == mla.MLA_ERR_INVALID_ARG
        assert call(y=None) == mla.MLA_ERR_INVALID_ARG
        assert call(w=0x10008) == mla.MLA_ERR_INVALID_ARG            # TMA needs 16-byte alignment
        assert call(x=0x20004) == mla.MLA_ERR_INVALID_ARG
        assert call(y=0x30001) == mla.MLA_ERR_INVALID_ARG            # bf16 output: 2-byte alignment
        assert call(n=65535 * 64 + 1) == mla.MLA_ERR_UNSUPPORTED     # grid z limit


def test_prefill_workspace_size_is_host_arithmetic(mla):
    # status header (256 B) + K^C and V, each T*H*128 bf16 rounded up to 256 B
    assert mla._lib.mla_prefill_workspace_size(4096, 128) == 256 + 2 * 4096 * 128 * 128 * 2
    assert mla._lib.mla_prefill_workspace_size(3, 2) == 256 + 2 * 1536
    assert mla._lib.mla_prefill_workspace_size(-1, 2) == 0
    assert mla._lib.mla_prefill_workspace_size(4, 0) == 0


def test_prefill_rejects_bad_arguments_before_launch(mla):
    import ctypes
    cc = mla.mla_cache_t(0x100000, 0x200000, mla.MLA_BF16, 2, 128, 64, 512, 64, 64)
    ws_need = mla._lib.mla_prefill_workspace_size(1000, 16)

    def call(cache=cc, seq=0, T=1000, H=16, scale=0.07, ws=0x400000, ws_bytes=ws_need, wk=0x500000, q=0x600000,
             out=0x700000):
        return mla._lib.mla_prefill_expanded(ctypes.byref(cache), seq, T, wk, wk, q, q, H, scale, out, None, ws,
                                             ws_bytes, None)

    assert call(T=0) == mla.MLA_OK                                   # empty: no launch
    assert call(seq=2) == mla.MLA_ERR_INVALID_ARG                    # beyond the page table's rows
    assert call(seq=-1) == mla.MLA_ERR_INVALID_ARG
    assert call(T=64 * 64 + 1) == mla.MLA_ERR_INVALID_ARG            # beyond the sequence's pages
    assert call(H=15) == mla.MLA_ERR_UNSUPPORTED                     # H even
    assert call(H=0) == mla.MLA_ERR_INVALID_ARG
    assert call(scale=0.0) == mla.MLA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == mla.MLA_ERR_INVALID_ARG
    assert call(ws=None) == mla.MLA_ERR_WORKSPACE
    assert call(ws=0x400010) == mla.MLA_ERR_WORKSPACE                # 256-byte alignment
    assert call(ws_bytes=ws_need - 1) == mla.MLA_ERR_WORKSPACE
    assert call(wk=None) == mla.MLA_ERR_INVALID_ARG
    assert call(q=0x600008) == mla.MLA_ERR_INVALID_ARG               # TMA needs 16-byte alignment
    assert call(out=None) == mla.MLA_ERR_INVALID_ARG
    fp32 = mla.mla_cache_t(0x100000, 0x200000, mla.MLA_FP32, 2, 128, 64, 64, 16, 64)
    assert call(cache=fp32) == mla.MLA_ERR_UNSUPPORTED               # bf16 cache only
