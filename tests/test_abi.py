"""The C-ABI library: builds for sm_103a, loads without a GPU, exports every
entry point include/attn.h declares, and rejects bad arguments on the host
before touching the device.  No compute call is made here."""
import ctypes
import os
import re

import pytest

import attention_attn_fwd_03_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    attn.build()
    return attn.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert _declared() == sorted(["attn_fwd", "attn_fwd_fp8", "attn_paged_decode",
                                  "attn_paged_decode_workspace_size", "attn_paged_decode_noalloc",
                                  "attn_paged_fwd", "attn_paged_fwd_workspace_size",
                                  "attn_varlen_fwd", "attn_varlen_fwd_workspace_size",
                                  "attn_bwd", "attn_bwd_workspace_size",
                                  "attn_fwd_host", "attn_fwd_host_workspace_size", "attn_selftest_wait_timeout",
                                  "attn_selftest_mma_rate", "attn_device_status", "attn_status_string"])


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
    raw = ctypes.CDLL(attn.LIB_PATH)
    for name in _declared():
        assert ctypes.cast(getattr(raw, name), ctypes.c_void_p).value


def test_status_strings(L):
    for code in range(7):
        s = attn.attn_status_string(code)
        assert s and s != "unknown status"
    assert attn.attn_status_string(99) == "unknown status"


FAKE = 1 << 20  # a 16-byte aligned non-NULL address; validation fails before any use


def _fwd(**kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, H=1, Nq=128, Nk=128, d=128, scale=0.088,
             causal=0, stream=None)
    a.update(kw)
    return attn.attn_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=None), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Nq=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Nk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), attn.ATTN_ERR_INVALID_ARG),
    (dict(lse=FAKE + 2), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
])
def test_fwd_validation(L, kw, code):
    assert _fwd(**kw) == code


def test_fp8_validation(L):
    base = dict(q8=FAKE, k8=FAKE, v8=FAKE, q_descale=1.0, k_descale=1.0, v_descale=1.0, o=FAKE, lse=None,
                B=1, H=1, Nq=64, Nk=64, d=128, scale=0.088, causal=0, stream=None)
    assert attn.attn_fwd_fp8(**dict(base, q_descale=0.0)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_fp8(**dict(base, v_descale=float("inf"))) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_fp8(**dict(base, d=64)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_fp8(**dict(base, k8=None)) == attn.ATTN_ERR_INVALID_ARG


def test_workspace_size_query(L):
    # argument order (B, H, d, max_pages_per_seq, page_size)
    ws = attn.attn_paged_decode_workspace_size(64, 32, 128, 128, 64)
    assert ws >= 64 * 32 * 130 * 4  # at least one (O, m, l) record per (request, head)
    assert attn.attn_paged_decode_workspace_size(64, 32, 128, 256, 64) > ws
    assert attn.attn_paged_decode_workspace_size(64, 32, 96, 128, 64) == 0
    assert attn.attn_paged_decode_workspace_size(64, 32, 128, 128, 12) == 0
    assert attn.attn_paged_decode_workspace_size(0, 32, 128, 128, 64) == 0
    # page_size is validated as a page size, max_pages_per_seq as a count:
    # 12 pages of 64 is valid, 64 pages of 12 is not
    assert attn.attn_paged_decode_workspace_size(64, 32, 128, 12, 64) > 0


def test_paged_decode_validation(L):
    ws = attn.attn_paged_decode_workspace_size(4, 2, 128, 8, 64)
    base = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, block_table=FAKE, seq_lens=FAKE, B=4, H=2, d=128,
                page_size=64, max_pages_per_seq=8, num_pages=32, scale=0.088, o=FAKE, lse=None,
                workspace=FAKE, workspace_bytes=ws, stream=None)
    assert attn.attn_paged_decode(**dict(base, workspace_bytes=ws - 1)) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_paged_decode(**dict(base, workspace=None)) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_paged_decode(**dict(base, page_size=12)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_paged_decode(**dict(base, d=80)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_paged_decode(**dict(base, seq_lens=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_decode(**dict(base, block_table=FAKE + 2)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_decode(**dict(base, num_pages=0)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_decode(**dict(base, scale=-1.0)) == attn.ATTN_ERR_INVALID_ARG


def test_library_has_no_oracle_dependency():
    """The product library links nothing from oracle/, and its sources name none of it."""
    csrc = os.path.join(ROOT, "attention_attn_fwd_03_gb300", "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        assert "oracle" not in text.lower(), f
    for f in ("__init__.py", "_build.py", "inputs.py"):
        text = open(os.path.join(ROOT, "attention_attn_fwd_03_gb300", f), encoding="utf-8").read()
        assert "import oracle" not in text and "from oracle" not in text, f


def test_paged_fwd_workspace_size_query(L):
    # one token per request over 8192-key caches: runs of 8 KV blocks, 8 splits
    ws = attn.attn_paged_fwd_workspace_size(64, 64, 1, 32, 8, 128, 64, 128)
    assert ws >= 64 * 32 * 8 * 130 * 4
    # everything fits one split: only the work list (8 entries of 16 bytes, rounded to 256) and its header
    assert attn.attn_paged_fwd_workspace_size(4, 4, 1, 8, 2, 128, 64, 16) == 512
    assert attn.attn_paged_fwd_workspace_size(4, 4, 1, 8, 3, 128, 64, 16) == 0  # H % H_kv != 0
    assert attn.attn_paged_fwd_workspace_size(4, 4, 1, 8, 2, 128, 48, 16) == 0  # page size not a power of two
    assert attn.attn_paged_fwd_workspace_size(4, 4, 1, 512, 2, 128, 64, 16) == 0  # 256 heads per group
    assert attn.attn_paged_fwd_workspace_size(4, 4, 5, 8, 2, 128, 64, 16) == 0  # max_q_len > total_q


def test_paged_fwd_validation(L):
    base = dict(q=FAKE, k_cache=FAKE, v_cache=FAKE, block_table=FAKE, cu_seqlens_q=None, seq_lens=FAKE, B=4,
                total_q=4, max_q_len=1, H=8, H_kv=2, d=128, page_size=64, max_pages_per_seq=16, num_pages=64,
                scale=0.088, causal=0, o=FAKE, lse=None, workspace=None, workspace_bytes=0, stream=None)
    assert attn.attn_paged_fwd(**dict(base, H_kv=3)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_fwd(**dict(base, total_q=5)) == attn.ATTN_ERR_INVALID_ARG  # no offsets: one token each
    assert attn.attn_paged_fwd(**dict(base, page_size=48)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_paged_fwd(**dict(base, d=96)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_paged_fwd(**dict(base, causal=2)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_fwd(**dict(base, q=FAKE + 8)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_fwd(**dict(base, num_pages=0)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_fwd(**dict(base, seq_lens=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_paged_fwd(**base) == attn.ATTN_ERR_WORKSPACE  # the work list is always needed
    long = dict(base, max_pages_per_seq=128, num_pages=1024)
    ws = attn.attn_paged_fwd_workspace_size(4, 4, 1, 8, 2, 128, 64, 128)
    assert ws > 0
    assert attn.attn_paged_fwd(**long) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_paged_fwd(**dict(long, workspace=FAKE, workspace_bytes=ws - 1)) == attn.ATTN_ERR_WORKSPACE


def test_varlen_fwd_validation(L):
    ws = attn.attn_varlen_fwd_workspace_size(4, 64, 32, 48, 8, 2, 128)
    assert ws > 0
    assert attn.attn_varlen_fwd_workspace_size(4, 64, 32, 0, 8, 2, 128) == 0
    assert attn.attn_varlen_fwd_workspace_size(4, 64, 32, 48, 8, 3, 128) == 0
    base = dict(q=FAKE, k=FAKE, v=FAKE, cu_seqlens_q=FAKE, cu_seqlens_k=FAKE, B=4, total_q=64, total_k=100,
                max_q_len=32, max_k_len=48, H=8, H_kv=2, d=128, scale=0.088, causal=1, o=FAKE, lse=None,
                workspace=FAKE, workspace_bytes=ws, stream=None)
    assert attn.attn_varlen_fwd(**dict(base, cu_seqlens_k=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_varlen_fwd(**dict(base, max_k_len=101)) == attn.ATTN_ERR_INVALID_ARG  # > total_k
    assert attn.attn_varlen_fwd(**dict(base, d=80)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_varlen_fwd(**dict(base, workspace_bytes=ws - 1)) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_varlen_fwd(**dict(base, cu_seqlens_q=FAKE + 2)) == attn.ATTN_ERR_INVALID_ARG


def test_paged_workspace_layout(L):
    """attn_paged_fwd's workspace: a 256-byte header, the unit list (16 bytes per unit, rounded to
    256), then for split launches the fp32 partial O and (m, l) per row and split, and for
    decode-like split launches one int per request (requests run unsplit)."""
    # 64 requests x 32 heads over 8 KV heads, one token each, up to 128 pages of 64 tokens:
    # 64 KV blocks per request in splits of 8 -> 8 splits, 64 * 8 * 8 units
    units = 64 * 8 * 8
    size = 256 + (units * 16 + 255) // 256 * 256
    size += 64 * 32 * 8 * 128 * 4          # partial O
    size += 64 * 32 * 8 * 2 * 4            # partial (m, l)
    size = (size + 255) // 256 * 256 + 64 * 4  # per-request flags
    assert attn.attn_paged_fwd_workspace_size(64, 64, 1, 32, 8, 128, 64, 128) == size
    # 8 KV blocks at most: one split, no partials, no flags
    assert attn.attn_paged_fwd_workspace_size(4, 4, 1, 8, 2, 128, 64, 16) == 256 + 256


def test_bwd_validation(L):
    ws = attn.attn_bwd_workspace_size(2, 4, 300, 128)
    assert ws == 2 * 4 * 384 * 130 * 4  # dQ accumulator + two row vectors, rows padded to 128
    assert attn.attn_bwd_workspace_size(2, 4, 300, 96) == 0
    base = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, B=2, H=4, Nq=300,
                Nk=300, d=128, scale=0.088, causal=1, workspace=FAKE, workspace_bytes=ws, stream=None)
    assert attn.attn_bwd(**dict(base, lse=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd(**dict(base, dk=FAKE + 8)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd(**dict(base, d=96)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_bwd(**dict(base, workspace_bytes=ws - 4)) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_bwd(**dict(base, causal=3)) == attn.ATTN_ERR_INVALID_ARG
    # (batch*head, 128-key block) units past 2^31: refused before anything is enqueued
    assert attn.attn_bwd(**dict(base, B=16, H=64, Nk=2 ** 30)) == attn.ATTN_ERR_UNSUPPORTED


def test_fwd_host_workspace_and_validation(L):
    """Slot sizes of the host-staged prefill (three slots, each rounded to 256-byte buffers) and the
    checks it makes before touching any device or host memory."""
    def r256(x):
        return (x + 255) // 256 * 256
    cb = 3
    slot = r256(cb * 300 * 128 * 2) + 2 * r256(cb * 200 * 128 * 2) + 2 * (r256(cb * 300 * 128 * 2) + r256(cb * 300 * 4))
    ws = attn.attn_fwd_host_workspace_size(2, 4, 300, 200, 128, 2, cb)
    assert ws == 3 * slot
    # default chunk: about an eighth of B*H (here one pair); a chunk larger than B*H is clipped to it
    assert attn.attn_fwd_host_workspace_size(2, 4, 300, 200, 128, 1, 0) == \
        attn.attn_fwd_host_workspace_size(2, 4, 300, 200, 128, 1, 1)
    assert attn.attn_fwd_host_workspace_size(2, 4, 300, 200, 128, 1, 100) == \
        attn.attn_fwd_host_workspace_size(2, 4, 300, 200, 128, 1, 8)
    for bad in [(2, 4, 300, 200, 96, 1, 1), (2, 4, 300, 200, 128, 0, 1), (2, 4, 300, 200, 128, 9, 1),
                (0, 4, 300, 200, 128, 1, 1), (2, 4, 0, 200, 128, 1, 1)]:
        assert attn.attn_fwd_host_workspace_size(*bad) == 0
    modes = (ctypes.c_int * 2)(0, 1)
    outs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    base = dict(q=FAKE, k=FAKE, v=FAKE, n_modes=2, causal=ctypes.addressof(modes), o=ctypes.addressof(outs),
                lse=None, B=2, H=4, Nq=300, Nk=200, d=128, scale=0.088, chunk_bh=cb, workspace=FAKE,
                workspace_bytes=ws, stream=None)
    assert attn.attn_fwd_host(**dict(base, v=None)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_host(**dict(base, n_modes=0)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_host(**dict(base, scale=-1.0)) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_host(**dict(base, d=96)) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_fwd_host(**dict(base, workspace_bytes=ws - 1)) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_fwd_host(**dict(base, workspace=FAKE + 4)) == attn.ATTN_ERR_WORKSPACE
    bad_modes = (ctypes.c_int * 2)(0, 2)
    assert attn.attn_fwd_host(**dict(base, causal=ctypes.addressof(bad_modes))) == attn.ATTN_ERR_INVALID_ARG
    no_out = (ctypes.c_void_p * 2)(FAKE, None)
    assert attn.attn_fwd_host(**dict(base, o=ctypes.addressof(no_out))) == attn.ATTN_ERR_INVALID_ARG


def test_noalloc_scratch_size_matches_header():
    """The binding's copy of ATTN_NOALLOC_SCRATCH_BYTES is the header's."""
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        m = re.search(r"#define ATTN_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", f.read())
    assert m is not None
    assert attn.ATTN_NOALLOC_SCRATCH_BYTES == int(m.group(1)) * int(m.group(2)) * int(m.group(3))


def test_selftest_mma_rate_validation(L):
    assert attn.attn_selftest_mma_rate(None, 1, 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_selftest_mma_rate(FAKE + 4, 1, 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_selftest_mma_rate(FAKE, 0, 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_selftest_mma_rate(FAKE, 1, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_selftest_mma_rate(FAKE, 1, (1 << 20) + 1, None) == attn.ATTN_ERR_INVALID_ARG
