"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/sagebwd.h declares, and rejects bad arguments before
any launch (those paths make no CUDA call)."""
import ctypes
import os
import re

import pytest

import bit_trainable_attention_gb300 as sb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sagebwd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(sagebwd_[a-z_0-9]+)\s*\(", text, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return sb.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("sagebwd_quantize", "sagebwd_fwd", "sagebwd_bwd", "sagebwd_check_status"):
        assert required in names
    assert set(names) == set(sb.EXPORTED_SYMBOLS)


def test_binding_constants_match_the_header():
    """The binding's copies of the header's flag and operand constants (the problem struct carries
    them as plain integers, so a mismatch would silently select another option)."""
    text = open(os.path.join(ROOT, "include", "sagebwd.h")).read()
    flags = {m[0]: int(m[1], 16) for m in re.findall(r"#define (SAGEBWD_FLAG_[A-Z0-9_]+) (0x[0-9a-fA-F]+)u", text)}
    assert flags["SAGEBWD_FLAG_DROP_ONE_LOAD"] == sb.FLAG_DROP_ONE_LOAD
    assert flags["SAGEBWD_FLAG_DEBUG_DUMP"] == sb.FLAG_DEBUG_DUMP
    for name, value in sb.FLAG_BF16.items():
        assert flags["SAGEBWD_FLAG_BF16_" + name.upper().replace("P_FWD", "PF").replace("P_BWD", "PB")] == value, name
    assert len({v for k, v in flags.items()}) == len(flags)  # no two flags share a bit pattern
    ops = dict(re.findall(r"(SAGEBWD_(?:Q|K|V|DO)) = (\d+)", text))
    assert {k: int(v) for k, v in ops.items()} == {"SAGEBWD_Q": sb.SAGEBWD_Q, "SAGEBWD_K": sb.SAGEBWD_K,
                                                   "SAGEBWD_V": sb.SAGEBWD_V, "SAGEBWD_DO": sb.SAGEBWD_DO}


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_sizes_and_strings(lib):
    p = sb.Problem.make(1, 4, 2, 300, 64, True)
    nb = 3
    saved = sb.sagebwd_saved_bytes(p)
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    expect = al(1 * 4 * 300 * 64 * 2) + 2 * al(1 * 2 * 300 * 64 * 2) + al(4 * nb * 4) + 2 * al(2 * nb * 4) + \
        2 * al(2 * 64 * 4)  # ... K mean, balancing exponents
    assert saved == expect
    assert sb.sagebwd_workspace_bytes(p, 0) >= 256 + 2 * nb * 64 * 8
    assert sb.sagebwd_workspace_bytes(p, 1) >= 256 + 4 * 300 * 64 * (4 + 2)
    assert sb.sagebwd_workspace_bytes(p, 2) == 0
    assert sb.sagebwd_status_string(0) == "ok"
    assert "timed out" in sb.sagebwd_status_string(5)
    assert sb.sagebwd_version() >= 100


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2),                    # unsupported head dim
    (dict(Hq=3, Hkv=2), 1),             # Hq % Hkv != 0
    (dict(N=0), 1),
    (dict(B=0), 1),
    (dict(N=1 << 30), 2),               # beyond int32 element indices
])
def test_bad_problems_rejected_before_launch(lib, kw, code):
    args = dict(B=1, Hq=4, Hkv=2, N=256, d=64, causal=True)
    args.update(kw)
    p = sb.Problem.make(**args)
    assert sb.sagebwd_saved_bytes(p) == 0
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    rc = lib.sagebwd_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, None)
    assert rc == code


def test_bad_pointers_rejected_before_launch(lib):
    p = sb.Problem.make(1, 4, 2, 256, 64, True)
    good = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.sagebwd_fwd(ctypes.byref(p), None, good, good, good, good, good, good, None) == 1
    assert lib.sagebwd_fwd(ctypes.byref(p), good, odd, good, good, good, good, good, None) == 3
    assert lib.sagebwd_bwd(ctypes.byref(p), *([good] * 5), odd, *([good] * 6)) == 3
    assert lib.sagebwd_quantize(ctypes.byref(p), 7, good, good, good, None, good, None) == 1
    # K with smoothing needs the mean output
    assert lib.sagebwd_quantize(ctypes.byref(p), 1, good, good, good, None, good, None) == 1
    assert lib.sagebwd_check_status(None, None, None) == 1


def test_balancing_sizes_and_rejections(lib):
    """With balance_qk the forward workspace adds the per-block channel maxima of K (max, min) and Q;
    the single-operand quantizers refuse Q and K (their codes would depend on both tensors)."""
    p0 = sb.Problem.make(1, 4, 2, 300, 64, True)
    p1 = sb.Problem.make(1, 4, 2, 300, 64, True, balance_qk=True)
    nb = 3
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert sb.sagebwd_saved_bytes(p1) == sb.sagebwd_saved_bytes(p0)
    extra = 2 * al(2 * nb * 64 * 4) + al(4 * nb * 64 * 4)
    assert sb.sagebwd_workspace_bytes(p1, 0) == sb.sagebwd_workspace_bytes(p0, 0) + extra
    assert sb.sagebwd_workspace_bytes(p1, 1) == sb.sagebwd_workspace_bytes(p0, 1)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls return before any launch
    for which in (sb.SAGEBWD_Q, sb.SAGEBWD_K):
        assert lib.sagebwd_quantize(ctypes.byref(p1), which, fake, fake, fake, fake, fake, None) == 2
    assert lib.sagebwd_quantize_k_noalloc(ctypes.byref(p1), fake, fake, fake, fake, None) == 2
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert lib.sagebwd_bwd_finish(ctypes.byref(p1), odd, fake, fake, fake, fake, None) == 3
    assert lib.sagebwd_bwd_finish(ctypes.byref(p1), None, fake, fake, fake, fake, None) == 1


def test_q_smoothing_sizes_and_rejections(lib):
    """With smooth_q the saved buffer adds the block means of Q and the logit terms, the backward
    workspace a ring of dS column sums per CTA; balancing together with it, and the single-operand
    quantizer for Q under it, are refused before any launch."""
    p0 = sb.Problem.make(2, 4, 2, 300, 64, True)
    p1 = sb.Problem.make(2, 4, 2, 300, 64, True, smooth_q=True)
    nb = 3
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert sb.sagebwd_saved_bytes(p1) == sb.sagebwd_saved_bytes(p0) + al(2 * 4 * nb * 64 * 4) + al(
        2 * 4 * nb * nb * 128 * 4)
    assert sb.sagebwd_workspace_bytes(p1, 0) == sb.sagebwd_workspace_bytes(p0, 0)
    assert sb.sagebwd_workspace_bytes(p1, 1) == sb.sagebwd_workspace_bytes(p0, 1) + al(2 * 4 * nb * 2 * 4 * 128 * 4)
    both = sb.Problem.make(2, 4, 2, 300, 64, True, smooth_q=True, balance_qk=True)
    assert sb.sagebwd_saved_bytes(both) == 0 and sb.sagebwd_workspace_bytes(both, 1) == 0
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls return before any launch
    assert lib.sagebwd_quantize(ctypes.byref(p1), sb.SAGEBWD_Q, fake, fake, fake, fake, fake, None) == 2
    assert lib.sagebwd_fwd(ctypes.byref(both), fake, fake, fake, fake, fake, fake, fake, None) == 2


def test_debug_dump_sizes_and_rejections(lib):
    """SAGEBWD_FLAG_DEBUG_DUMP adds one record per tile to each workspace (forward 128*128*6 + 512 d
    bytes, backward 65536 + 1536 d bytes), with the Q/K sub-scales (the default) or without, and is
    refused with the dS sub-scales and Q-smoothing (other kernel instantiations)."""
    p0 = sb.Problem.make(1, 2, 1, 300, 64, True)
    p1 = sb.Problem.make(1, 2, 1, 300, 64, True, flags=sb.FLAG_DEBUG_DUMP)
    nb = 3
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert sb.sagebwd_workspace_bytes(p1, 0) == sb.sagebwd_workspace_bytes(p0, 0) + al(2 * nb * nb * (98304 + 512 * 64))
    assert sb.sagebwd_workspace_bytes(p1, 1) == sb.sagebwd_workspace_bytes(p0, 1) + al(2 * nb * nb * (65536 + 1536 * 64))
    assert sb.sagebwd_debug_dump_offset(p0, 0) == 0 and sb.sagebwd_debug_dump_offset(p1, 1) > 0
    assert sb.sagebwd_debug_dump_offset(p1, 0) + al(2 * nb * nb * (98304 + 512 * 64)) == sb.sagebwd_workspace_bytes(p1, 0)
    plain = sb.Problem.make(1, 2, 1, 300, 64, True, flags=sb.FLAG_DEBUG_DUMP, qk_subexp=False)
    assert sb.sagebwd_workspace_bytes(plain, 1) == sb.sagebwd_workspace_bytes(p1, 1)
    for opt in ("ds_subexp", "smooth_q"):
        bad = sb.Problem.make(1, 2, 1, 300, 64, True, flags=sb.FLAG_DEBUG_DUMP, **{opt: True})
        assert sb.sagebwd_workspace_bytes(bad, 1) == 0, opt
    huge = sb.Problem.make(1, 32, 8, 65536, 128, False, flags=sb.FLAG_DEBUG_DUMP)
    assert sb.sagebwd_saved_bytes(huge) == 0


def test_attribution_flags_refused_with_unsupported_options(lib):
    """The BF16 attribution flags cover the kernels without dS sub-scales, Q-smoothing and the dump."""
    ok = sb.Problem.make(1, 2, 1, 300, 64, True, flags=sb.FLAG_BF16["ds"] | sb.FLAG_BF16["q"])
    assert sb.sagebwd_workspace_bytes(ok, 1) > 0
    for opts, flags in (({"ds_subexp": True}, 0), ({"smooth_q": True}, 0), ({}, sb.FLAG_DEBUG_DUMP)):
        p = sb.Problem.make(1, 2, 1, 300, 64, True, flags=sb.FLAG_BF16["ds"] | flags, **opts)
        assert sb.sagebwd_workspace_bytes(p, 1) == 0, opts


def test_fp8_variant_sizes_and_refusals(lib):
    """The FP8 variant keeps the INT8 layouts (E4M3 values held in the same BF16 buffers), adds the same
    values as bytes (Q, K [BH][N][d], V transposed per head [BHk][d][128 nb]) and refuses the INT8-only
    refinements."""
    p8 = sb.Problem.make(1, 4, 2, 300, 64, True, fp8=True)
    assert p8.qk_subexp == 0  # no sub-scales for E4M3 values
    p0 = sb.Problem.make(1, 4, 2, 300, 64, True, qk_subexp=False)
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    extra = al(4 * 300 * 64) + al(2 * 300 * 64) + al(2 * 64 * 3 * 128)
    assert sb.sagebwd_saved_bytes(p8) == sb.sagebwd_saved_bytes(p0) + extra > 0
    assert sb.sagebwd_workspace_bytes(p8, 1) == sb.sagebwd_workspace_bytes(p0, 1)
    for opts in ({"qk_subexp": True}, {"ds_subexp": True}, {"balance_qk": True}, {"smooth_q": True},
                 {"flags": sb.FLAG_BF16["ds"]}, {"flags": sb.FLAG_DEBUG_DUMP}):
        assert sb.sagebwd_saved_bytes(sb.Problem.make(1, 4, 2, 300, 64, True, fp8=True, **opts)) == 0, opts
