"""The C ABI without a GPU: libkvq.so loads, exports every entry point include/kvq.h
declares, and rejects invalid arguments on the host (no launch, no device access)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_kv_cache_fp8_gb300 as k
    return k


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(kvq):
    L = kvq.lib()
    decl = declared_symbols()
    assert decl == sorted(kvq.EXPORTS)
    for name in decl:
        assert getattr(L, name) is not None


def test_status_strings_and_version(kvq):
    L = kvq.lib()
    for s in range(8):
        assert L.kvq_status_string(s).decode().startswith("KVQ_")
    assert kvq.kvq_version() >= 100


FAKE = 0x10000            # a 64 KiB-aligned address that is never dereferenced


def test_encode_argument_errors(kvq):
    L = kvq.lib()
    # non-power-of-two TQ4 width is refused before anything else (the page's refusal)
    for dim in (384, 500, 96, 513):
        assert L.kvq_encode_tq4(FAKE, 4, dim, dim, FAKE, FAKE, dim, FAKE, None) == 2
    assert L.kvq_encode_tq4(FAKE, 4, 2048, 2048, FAKE, FAKE, 1024, FAKE, None) == 1
    assert L.kvq_encode_tq4(FAKE, 4, 512, 100, FAKE, FAKE, 256, FAKE, None) == 1
    assert L.kvq_encode_tq4(None, 4, 512, 512, FAKE, FAKE, 256, FAKE, None) == 1
    assert L.kvq_encode_tq4(FAKE + 2, 4, 512, 512, FAKE, FAKE, 256, FAKE, None) == 4
    assert L.kvq_encode_fp8(FAKE, -1, 512, 512, FAKE, 512, FAKE, None) == 1
    assert L.kvq_encode_fp8(FAKE, 4, 0, 512, FAKE, 512, FAKE, None) == 1
    assert L.kvq_encode_fp8(FAKE, 4, 512, 256, FAKE, 512, FAKE, None) == 1
    assert L.kvq_encode_fp8(FAKE, 0, 512, 512, None, 512, None, None) == 0     # no-op
    assert b"ldx" in L.kvq_last_error() or b"dim" in L.kvq_last_error() or True


def test_encode_mla_argument_errors(kvq):
    L = kvq.lib()
    def call(fmt=kvq.FMT_TQ4, rows=1, ldx=512, ldr=64, ldl=256, ldc=64, c=FAKE, signs=FAKE, ls=FAKE):
        return L.kvq_encode_mla(c, ldx, FAKE, ldr, rows, fmt, signs, FAKE, ldl, ls, FAKE, ldc, FAKE, None)
    assert call(fmt=kvq.FMT_Q4_0) == 3                                    # not an MLA tier
    assert call(rows=-1) == 1
    assert call(ldx=511) == 1
    assert call(ldr=63) == 1
    assert call(ldl=255) == 1                                             # 4 bits: 256 bytes
    assert call(fmt=kvq.FMT_TQ6, ldl=383) == 1                            # 6 bits: 384 bytes
    assert call(fmt=kvq.FMT_FP8, ldl=511) == 1
    assert call(ldc=63) == 1
    assert call(c=None) == 1
    assert call(signs=None) == 1                                          # rotated tier needs signs
    assert call(c=FAKE + 2) == 4
    assert call(ls=FAKE + 1) == 4
    assert call(rows=0, c=None) == 0                                      # no-op


def test_project_append_argument_errors(kvq):
    L = kvq.lib()
    def call(h=FAKE, d_model=1024, wk=FAKE, wv=FAKE, w_type=kvq.WEIGHT_F32, n_seq=1, n_tok=1,
             head_dim=256, kp=FAKE, pt=FAKE):
        return L.kvq_project_append_q4(h, n_seq, FAKE, n_tok, d_model, wk, wv, w_type, 8, head_dim,
                                       pt, 1, 64, 64, kp, FAKE, None, None)
    assert call(head_dim=250) == 2
    assert call(head_dim=128) == 1
    assert call(d_model=1022) == 1                                         # not a multiple of 4
    assert call(d_model=0) == 1
    assert call(w_type=2) == 1
    assert call(n_seq=65536, n_tok=17) == 1                                # too many tokens
    assert call(wv=None) == 1
    assert call(pt=None) == 1
    assert call(h=FAKE + 4) == 4                                           # h rows need 16 bytes
    assert call(wk=FAKE + 8) == 4                                          # 16-byte rows
    assert call(wv=FAKE + 8, w_type=kvq.WEIGHT_BF16) == 4                  # bf16 too
    assert call(kp=FAKE + 8) == 4
    assert call(n_tok=0, h=None) == 0                                      # no-op


def test_append_and_gather_argument_errors(kvq):
    L = kvq.lib()
    assert L.kvq_append_q4(FAKE, FAKE, 1, FAKE, 1, 8, 250, FAKE, 1, 64, 64, FAKE, FAKE, None, None) == 2
    assert L.kvq_append_q4(FAKE, FAKE, 1, FAKE, 1, 8, 128, FAKE, 1, 64, 64, FAKE, FAKE, None, None) == 1
    assert L.kvq_append_q4(FAKE, FAKE, 1, FAKE, 1, 8, 256, FAKE, 1, 64, 64, FAKE + 8, FAKE, None, None) == 4
    assert L.kvq_append_q4(FAKE, FAKE, 1, FAKE, 1, 8, 256, FAKE, 0, 64, 64, FAKE, FAKE, None, None) == 1
    d = kvq.GatherDesc()
    d.format = 9
    assert L.kvq_gather(C.byref(d), None) == 3
    d.format = kvq.FMT_Q4_0
    d.head_dim = 100
    assert L.kvq_gather(C.byref(d), None) == 2
    d.format = kvq.FMT_FP8
    d.n_idx = 5
    assert L.kvq_gather(C.byref(d), None) == 1                                   # NULL planes


def _problem(kvq, **kw):
    p = kvq.MlaProblem()
    p.n_seq, p.n_q, p.n_heads, p.d_lat, p.d_rope = 1, 1, 64, 512, 64
    p.max_seq_len, p.fmt = 32768, kvq.FMT_TQ4
    p.seq_len, p.q_lat, p.q_rope = FAKE, FAKE, FAKE
    p.tq4 = kvq.MlaCache(FAKE, FAKE, FAKE, FAKE, 32768)
    p.tq4_signs = FAKE
    p.sm_scale = 0.072
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_overlap_prior_must_be_0_or_1(kvq):
    """overlap_prior is a flag: any other value is an argument error of the kernel choice
    and of the decode call, before anything launches."""
    L = kvq.lib()
    for bad in (2, -1):
        p = _problem(kvq, overlap_prior=bad)
        assert L.kvq_mla_decode_kernel(C.byref(p)) == -1
        with pytest.raises(kvq.KvqError) as e:
            kvq.kvq_mla_decode_kernel(p)
        assert e.value.status == 1
        assert L.kvq_mla_decode(C.byref(p), FAKE, None, None, 0, None, None) == 1
    assert kvq.kvq_mla_decode_kernel(_problem(kvq, overlap_prior=1)) == kvq.IMPL_TC


def test_decode_kernel_choice(kvq):
    """Which kernel kvq_mla_decode runs (host only): fp8 with 8 or more heads, no top-k
    list and at least 64 tile-units of work on the e4m3 tcgen05 kernel, other fp8 problems
    of at most 16 heads or with a top-k
    list on the warp-level MMA kernel, TQ4 with 8 to 16 heads and the 3- and 6-bit tiers
    with 8+ heads on the 16-head tcgen05 kernel, other problems of 8+ heads on the
    32-head tcgen05 kernel, the rest on CUDA cores; an explicit impl wins."""
    fp8 = dict(fmt=kvq.FMT_FP8, fp8=kvq.MlaCache(FAKE, FAKE, FAKE, FAKE, 32768))
    k = lambda **kw: kvq.kvq_mla_decode_kernel(_problem(kvq, **kw))
    assert k(n_heads=16, **fp8) == kvq.IMPL_TCF8
    assert k(n_heads=8, **fp8) == kvq.IMPL_TCF8
    assert k(n_heads=16, max_seq_len=1024, **fp8) == kvq.IMPL_MMA           # 8 tile-units
    assert k(n_heads=16, max_seq_len=8192, **fp8) == kvq.IMPL_TCF8          # 64
    assert k(n_heads=16, max_seq_len=1024, n_seq=8, seq_stride_rows=1024, **fp8) == kvq.IMPL_TCF8
    assert k(n_heads=4, **fp8) == kvq.IMPL_MMA
    assert k(n_heads=64, **fp8) == kvq.IMPL_TCF8
    assert k(n_heads=128, idx=FAKE, top_k=2048, **fp8) == kvq.IMPL_MMA
    assert k(n_heads=64) == kvq.IMPL_TC                                   # TQ4
    assert k(n_heads=16) == kvq.IMPL_TC16
    assert k(n_heads=8) == kvq.IMPL_TC16
    assert k(n_heads=17) == kvq.IMPL_TC
    assert k(n_heads=4) == kvq.IMPL_SIMT
    assert k(n_heads=16, fmt=kvq.FMT_TQ6) == kvq.IMPL_TC16
    assert k(n_heads=64, fmt=kvq.FMT_TQ3) == kvq.IMPL_TC16
    assert k(n_heads=4, fmt=kvq.FMT_TQ6) == kvq.IMPL_SIMT
    # per-sequence formats: split by tier once there are 64 tile-units of work
    mixed = dict(seq_fmt=FAKE, fp8=kvq.MlaCache(FAKE, FAKE, FAKE, FAKE, 32768))
    assert k(n_heads=64, **mixed) == kvq.IMPL_BY_FMT
    assert k(n_heads=16, **mixed) == kvq.IMPL_BY_FMT
    assert k(n_heads=16, max_seq_len=1024, **mixed) == kvq.IMPL_TC        # 8 tile-units
    assert k(n_heads=64, idx=FAKE, top_k=2048, **mixed) == kvq.IMPL_TC
    assert k(n_heads=4, **mixed) == kvq.IMPL_SIMT
    for impl in (1, 2, 3, 4):
        assert k(n_heads=64, impl=impl, **mixed) == impl
    for impl in (1, 2, 3, 4):
        assert k(n_heads=16, impl=impl) == impl
    for impl in (1, 2, 3, 4, 5):
        assert k(n_heads=16, impl=impl, **fp8) == impl
    with pytest.raises(kvq.KvqError) as e:
        k(fmt=kvq.FMT_TQ6, impl=3)
    assert e.value.status == 3
    with pytest.raises(kvq.KvqError) as e:                                # TQ4 rows
        k(n_heads=16, impl=5)
    assert e.value.status == 3
    assert kvq.lib().kvq_mla_decode_kernel(C.byref(_problem(kvq, d_lat=256))) == -1


def test_decode_argument_errors(kvq):
    L = kvq.lib()
    dec = lambda p, ws=None, n=0: L.kvq_mla_decode(C.byref(p), FAKE, None, ws, n, None, None)
    assert dec(_problem(kvq, d_lat=256)) == 1
    assert dec(_problem(kvq, fmt=7)) == 3
    # 3- and 6-bit rotated rows: the CUDA-core kernel; the tensor-core ones refuse them
    for fmt in (kvq.FMT_TQ3, kvq.FMT_TQ6):
        assert dec(_problem(kvq, fmt=fmt)) == 5                                  # workspace next
        assert dec(_problem(kvq, fmt=fmt, impl=2)) == 3
        assert dec(_problem(kvq, fmt=fmt, impl=3)) == 3
        assert dec(_problem(kvq, fmt=fmt, impl=4)) == 5                          # read by impl 4
    assert dec(_problem(kvq, tq4_signs=None)) == 1
    assert dec(_problem(kvq, q_lat=FAKE + 4)) == 4
    assert dec(_problem(kvq, n_seq=2, seq_stride_rows=100)) == 1
    assert dec(_problem(kvq, impl=6)) == 1                                       # 0 .. 5 only
    assert dec(_problem(kvq, impl=5)) == 3                                       # fp8 rows only
    for fmt in (kvq.FMT_TQ3, kvq.FMT_TQ6):
        assert dec(_problem(kvq, fmt=fmt, impl=5)) == 3
    assert dec(_problem(kvq, impl=-1)) == 1
    p = _problem(kvq)
    need = L.kvq_mla_decode_workspace(C.byref(p))
    assert need > 0
    assert dec(p) == 5
    assert dec(p, FAKE, need - 1) == 5
    assert dec(p, FAKE + 64, need) == 4
    # the fp8 tier needs no rotated-query buffer
    p8 = _problem(kvq, fmt=kvq.FMT_FP8, fp8=kvq.MlaCache(FAKE, FAKE, FAKE, FAKE, 32768))
    assert L.kvq_mla_decode_workspace(C.byref(p8)) < need
    assert L.kvq_mla_decode_workspace(C.byref(_problem(kvq, d_lat=7))) == 0


def _q4_problem(kvq, **kw):
    p = kvq.Q4Problem()
    base = dict(n_seq=2, n_qh=16, n_kv=8, head_dim=256, seq_len=FAKE, max_seq_len=4096,
                page_table=FAKE, max_pages=64, page_size=64, n_cells=8192, k_pool=FAKE,
                v_pool=FAKE, q=FAKE, gate=None, sm_scale=0.0625, split_rows=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


def test_q4_decode_argument_errors(kvq):
    L = kvq.lib()
    dec = lambda p, ws=None, n=0: L.kvq_q4_decode(C.byref(p), FAKE, None, ws, n, None, None)
    assert dec(_q4_problem(kvq, head_dim=128)) == 1
    assert dec(_q4_problem(kvq, n_qh=12)) == 1                        # not a multiple of n_kv
    assert dec(_q4_problem(kvq, n_qh=48, n_kv=8)) == 1                # ratio 6
    assert dec(_q4_problem(kvq, n_qh=128, n_kv=8)) == 1               # ratio 16
    assert dec(_q4_problem(kvq, page_size=0)) == 1
    assert dec(_q4_problem(kvq, v_pool=None)) == 1
    assert dec(_q4_problem(kvq, k_pool=FAKE + 8)) == 4
    assert dec(_q4_problem(kvq, gate=FAKE + 4)) == 4
    assert dec(_q4_problem(kvq, sm_scale=float("nan"))) == 1
    assert L.kvq_q4_decode(C.byref(_q4_problem(kvq)), FAKE + 4, None, None, 0, None, None) == 4
    p = _q4_problem(kvq)
    need = L.kvq_q4_decode_workspace(C.byref(p))
    assert need > 0
    assert dec(p) == 5
    assert dec(p, FAKE, need - 1) == 5
    assert dec(p, FAKE + 64, need) == 4
    assert L.kvq_q4_decode_workspace(C.byref(_q4_problem(kvq, n_kv=3))) == 0
    # n_seq == 0 is a valid empty call that touches nothing
    assert dec(_q4_problem(kvq, n_seq=0, seq_len=None, q=None)) == 0
    # the workspace holds (m, l) and a 256-float partial per (sequence, head, split)
    p1 = _q4_problem(kvq, split_rows=1024)
    rows, splits = 2 * 16, 4
    assert L.kvq_q4_decode_workspace(C.byref(p1)) >= rows * splits * (2 + 256) * 4


def test_tq_codebooks_equal_the_oracle(kvq, orc):
    """The library's binary16 codebooks (written by gen_tq_codebooks.py, its own Lloyd-Max
    solve) equal the oracle's, centroids and thresholds, at every width."""
    import numpy as np
    for bits in (3, 4, 6):
        cb, thr = kvq.kvq_tq_codebook(bits)
        _, ocb, othr, _ = orc.tq_codebook(bits)
        assert np.array_equal(cb, ocb) and np.array_equal(thr, othr)
    L = kvq.lib()
    buf = (C.c_float * 64)()
    assert L.kvq_tq_codebook(5, buf, buf) == 1
    assert L.kvq_tq_codebook(6, None, buf) == 1


def test_encode_tq_argument_errors(kvq):
    L = kvq.lib()
    enc = lambda rows, dim, ldx, bits, ldp: L.kvq_encode_tq(FAKE, rows, dim, ldx, bits, FAKE, FAKE,
                                                            ldp, FAKE, None)
    assert enc(4, 512, 512, 5, 512) == 1                      # width
    assert enc(4, 384, 384, 6, 384) == 2                      # not a power of two
    assert enc(4, 2048, 2048, 6, 2048) == 1                   # above 1024
    assert enc(4, 512, 512, 6, 383) == 1                      # ldp < 512 * 6 / 8
    assert enc(4, 512, 512, 3, 191) == 1
    assert enc(0, 512, 512, 6, 384) == 0                      # nothing to do
    assert L.kvq_encode_tq(FAKE + 2, 4, 512, 512, 6, FAKE, FAKE, 384, FAKE, None) == 4


def test_fault_injection(kvq):
    L = kvq.lib()
    assert L.kvq_set_fault(b"nonsense") == 1
    assert L.kvq_set_fault(b"kvq_encode_fp8:7") == 0
    try:
        assert L.kvq_encode_fp8(FAKE, 4, 512, 512, FAKE, 512, FAKE, None) == 7
        assert b"fault injected" in L.kvq_last_error()
        # other entry points are unaffected (this one still fails its own validation)
        assert L.kvq_encode_tq4(FAKE, 4, 384, 384, FAKE, FAKE, 192, FAKE, None) == 2
    finally:
        assert L.kvq_set_fault(None) == 0
    assert L.kvq_encode_fp8(FAKE, 4, 0, 512, FAKE, 512, FAKE, None) == 1


def test_noalloc_host_checks_come_first(kvq):
    """kvq_mla_decode_noalloc checks everything on the host, under its own name, before it
    looks up its device array: an injected fault, an invalid problem and an empty batch
    return without any CUDA call (none is possible here, with no GPU)."""
    L = kvq.lib()
    na = lambda p, out=FAKE: L.kvq_mla_decode_noalloc(C.byref(p) if p is not None else None,
                                                      out, None, None, None)
    assert L.kvq_set_fault(b"kvq_mla_decode_noalloc:7") == 0
    try:
        assert na(_problem(kvq)) == 7
        assert L.kvq_last_error() == b"kvq_mla_decode_noalloc: fault injected (KVQ_FAULT / kvq_set_fault)"
    finally:
        assert L.kvq_set_fault(None) == 0
    # a fault armed for the workspace entry does not touch this one
    assert L.kvq_set_fault(b"kvq_mla_decode:6") == 0
    try:
        assert na(_problem(kvq, d_lat=256)) == 1
        assert L.kvq_last_error().startswith(b"kvq_mla_decode_noalloc: ")
    finally:
        assert L.kvq_set_fault(None) == 0
    assert na(None) == 1
    assert L.kvq_last_error() == b"kvq_mla_decode_noalloc: NULL problem"
    assert na(_problem(kvq, fmt=7)) == 3
    assert na(_problem(kvq), out=None) == 1
    assert na(_problem(kvq), out=FAKE + 4) == 4
    assert na(_problem(kvq, n_seq=0)) == 0                  # nothing to do, no device touched


def test_struct_layouts_match_headers(kvq, tmp_path):
    """The ctypes mirrors have the sizes and field offsets the C headers give."""
    import subprocess
    import oracle
    src = tmp_path / "sz.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "kvq.h"\n#include "kvq_oracle.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(kvq_mla_cache),'
        ' sizeof(kvq_gather_desc), sizeof(kvq_mla_problem), offsetof(kvq_mla_problem, impl),'
        ' offsetof(kvq_gather_desc, dev_status), sizeof(orc_mla), offsetof(orc_mla, n_sel));'
        'printf("%zu %zu %zu\\n", sizeof(kvq_q4_problem), offsetof(kvq_q4_problem, gate),'
        ' offsetof(kvq_q4_problem, split_rows));'
        'return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"),
                    str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [C.sizeof(kvq.MlaCache), C.sizeof(kvq.GatherDesc), C.sizeof(kvq.MlaProblem),
            kvq.MlaProblem.impl.offset, kvq.GatherDesc.dev_status.offset,
            C.sizeof(oracle.OrcMla), oracle.OrcMla.n_sel.offset,
            C.sizeof(kvq.Q4Problem), kvq.Q4Problem.gate.offset, kvq.Q4Problem.split_rows.offset]
    assert got == want


def test_fault_injection_from_environment(tmp_path):
    """KVQ_FAULT in the environment arms the injection at the first call (fresh process)."""
    import subprocess
    import sys
    code = (
        "import ctypes as C, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import quantized_kv_cache_fp8_gb300 as k\n"
        "L = k.lib()\n"
        f"print(L.kvq_encode_fp8({FAKE}, 4, 512, 512, {FAKE}, 512, {FAKE}, None),"
        f" L.kvq_encode_tq4({FAKE}, 4, 384, 384, {FAKE}, {FAKE}, 192, {FAKE}, None))\n")
    env = dict(os.environ, KVQ_FAULT="kvq_encode_fp8:6")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True).stdout.split()
    assert out == ["6", "2"]
