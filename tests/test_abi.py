"""The C-ABI library on the CPU: it builds, loads, exports every entry point
that include/pa.h declares, and its host-only logic (status names, workspace
size, partition plan, argument checks that return before any CUDA call)
behaves as documented.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_varlen_gb300 import build
    from paged_kv_varlen_gb300 import binding
    build.build_library()
    return binding.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_three_hot_path_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_varlen_attention", "pa_split_kv_reduce"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings_and_build_info(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(3) == b"PA_ERR_WORKSPACE"
    assert b"sm_103a" in lib.pa_build_info()


def test_workspace_size(lib):
    # the multi-query kernel's unit plan comes first: 4 header ints, then
    # order[S] and P[S + 1] (ints), rounded up to 256 bytes
    plan = (4 + 2 * 4 + 1) * 4
    plan = (plan + 255) // 256 * 256
    # forced P = 512: 4 seqs x ceil(8192/512)=16 parts x 32 heads x (128 + 2) floats
    # plus one extra partial slot (8 heads x (128 + 2) floats) per decode CTA
    # (256 at most) for items cut between CTAs, and their 16-byte table entries
    n = lib.pa_varlen_attention_workspace_size(4, 8192, 32, 128, 512)
    units = 4 * 16 * 32
    extra = 256 * 8 * (128 + 2) * 4 + 256 * 16
    assert n >= plan + units * (128 + 2) * 4 + extra
    assert n < plan + units * (128 + 2) * 4 + extra + 6 * 256
    # no split: the plan alone
    assert lib.pa_varlen_attention_workspace_size(4, 8192, 32, 128, -1) == plan
    big = lib.pa_varlen_attention_workspace_size(65535, 0, 32, 128, -1)
    assert big == ((4 + 2 * 65535 + 1) * 4 + 255) // 256 * 256
    # auto is bounded by the smallest partition it may choose (256)
    assert (lib.pa_varlen_attention_workspace_size(4, 8192, 32, 128, 0)
            >= lib.pa_varlen_attention_workspace_size(4, 8192, 32, 128, 256))


def test_partition_plan(lib):
    f = lib.pa_choose_partition_size
    assert f(32, 8, 8193, -1, 152) == 0         # never split
    assert f(32, 8, 8193, 512, 152) == 512      # forced
    assert f(32, 8, 300, 0, 152) == 0           # short contexts: no split
    assert f(32, 8, 8192, 0, 152) == 1024       # plenty of work: long partitions
    assert f(16, 8, 4096, 0, 152) == 512        # enough work with 512-key partitions
    assert f(2, 4, 65536, 0, 152) in (256, 512)
    assert f(1, 1, 4096, 0, 152) == 256         # tiny batch: shorter partitions


def _call_attention(lib, **over):
    args = dict(out=16, q=16, kc=16, vc=16, cu=16, sl=16, bt=16, mbps=4, S=2, total_q=2,
                mq=1, mk=40, Hq=4, Hkv=2, D=64, bs=16, nb=16, scale=0.125, sinks=None,
                causal=1, P=0, ws=None, ws_bytes=0, dtype=0, stream=None)
    args.update(over)
    v = ctypes.c_void_p
    return lib.pa_varlen_attention(
        v(args["out"]), v(args["q"]), v(args["kc"]), v(args["vc"]), v(args["cu"]), v(args["sl"]),
        v(args["bt"]), args["mbps"], args["S"], args["total_q"], args["mq"], args["mk"],
        args["Hq"], args["Hkv"], args["D"], args["bs"], args["nb"], args["scale"],
        args["sinks"], args["causal"], args["P"], args["ws"], args["ws_bytes"], args["dtype"],
        args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(out=0), 1),                 # null output
    (dict(dtype=7), 1),               # unknown dtype
    (dict(Hq=5), 1),                  # H_q not a multiple of H_kv
    (dict(Hq=18, Hkv=2), 2),          # group of 9 > 8
    (dict(D=96), 2),                  # head_dim not compiled
    (dict(bs=12), 2),                 # block size not a multiple of 8
    (dict(P=100), 1),                 # partition not a multiple of 32
    (dict(q=24), 1),                  # misaligned query pointer
    (dict(S=0), 1),                   # rows without requests
    (dict(total_q=0), 0),             # nothing to do
])
def test_attention_argument_checks_return_before_any_launch(lib, over, status):
    assert _call_attention(lib, **over) == status


def _call_scatter_and_attend(lib, **over):
    args = dict(key=16, value=16, stride=128, slots=16, T=2, out=16, q=16, kc=16, vc=16, cu=16,
                sl=16, bt=16, mbps=4, S=2, total_q=2, mq=1, mk=40, Hq=4, Hkv=2, D=64, bs=16,
                nb=16, scale=0.125, sinks=None, causal=1, P=0, ws=None, ws_bytes=0, dtype=0,
                stream=None)
    args.update(over)
    v = ctypes.c_void_p
    return lib.pa_scatter_and_attend(
        v(args["key"]), v(args["value"]), args["stride"], v(args["slots"]), args["T"],
        v(args["out"]), v(args["q"]), v(args["kc"]), v(args["vc"]), v(args["cu"]), v(args["sl"]),
        v(args["bt"]), args["mbps"], args["S"], args["total_q"], args["mq"], args["mk"],
        args["Hq"], args["Hkv"], args["D"], args["bs"], args["nb"], args["scale"],
        args["sinks"], args["causal"], args["P"], args["ws"], args["ws_bytes"], args["dtype"],
        args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(T=3), 1),                    # one new K/V row per query row
    (dict(stride=100), 1),             # token stride < H_kv * D
    (dict(key=0), 1),                  # null key rows
    (dict(slots=0), 1),                # null slot mapping
    (dict(key=17, dtype=1), 1),        # bf16 key rows not 2-byte aligned
    (dict(dtype=5), 1),                # unknown dtype
    (dict(Hq=18, Hkv=2, stride=256), 2),   # the attention's own checks follow: group of 9
    (dict(D=96, stride=192), 2),       # head_dim not compiled
    (dict(T=0, total_q=0), 0),         # nothing to do
])
def test_scatter_and_attend_argument_checks(lib, over, status):
    """The step call checks its scatter arguments, then the attention's, all
    before any CUDA call."""
    assert _call_scatter_and_attend(lib, **over) == status


def test_static_scratch_with_no_rows_needs_no_device(lib):
    """No rows: PA_OK (or the dtype error) before any device query, as for
    pa_varlen_attention itself."""
    v = ctypes.c_void_p
    f = lib.pa_varlen_attention_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, v, v, v, v, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_float, v, ctypes.c_int, ctypes.c_int, ctypes.c_int, v]
    base = [v(16)] * 7 + [4, 2, 0, 1, 40, 4, 2, 64, 16, 16, 0.125, None, 1, 0]
    assert f(*base, 0, None) == 0
    assert f(*base, 7, None) == 1


@pytest.mark.parametrize("over,status", [
    (dict(dtype=7), 1),               # unknown dtype
    (dict(out=0), 1),                 # null output
    (dict(q=24), 1),                  # misaligned query pointer
    (dict(P=100), 1),                 # partition not a multiple of 32
    (dict(P=-5), 1),                  # partition below -1
    (dict(D=96), 2),                  # head_dim not compiled
    (dict(Hq=72, Hkv=8), 2),          # group of 9 > 8
])
def test_static_scratch_checks_arguments_like_the_workspace_call(lib, over, status):
    """A bad argument gets the same status and message from the allocation-free
    call as from pa_varlen_attention, even when the split plan would need far
    more than the static array (64 requests of 64k keys), and before any device
    query (these run without a GPU)."""
    v = ctypes.c_void_p
    f = lib.pa_varlen_attention_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, v, v, v, v, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_float, v, ctypes.c_int, ctypes.c_int, ctypes.c_int, v]
    a = dict(out=16, q=16, kc=16, vc=16, cu=16, sl=16, bt=16, mbps=4096, S=64, total_q=64,
             mq=1, mk=65536, Hq=32, Hkv=8, D=128, bs=16, nb=4096, scale=0.1, sinks=None,
             causal=1, P=256, dtype=1)
    a.update(over)
    got = f(v(a["out"]), v(a["q"]), v(a["kc"]), v(a["vc"]), v(a["cu"]), v(a["sl"]), v(a["bt"]),
            a["mbps"], a["S"], a["total_q"], a["mq"], a["mk"], a["Hq"], a["Hkv"], a["D"], a["bs"],
            a["nb"], a["scale"], a["sinks"], a["causal"], a["P"], a["dtype"], None)
    msg = lib.pa_last_error_string().decode()
    assert got == status
    ref = _call_attention(lib, out=a["out"], q=a["q"], mbps=a["mbps"], S=a["S"],
                          total_q=a["total_q"], mk=a["mk"], Hq=a["Hq"], Hkv=a["Hkv"], D=a["D"],
                          nb=a["nb"], P=a["P"], dtype=a["dtype"])
    assert ref == status
    assert lib.pa_last_error_string().decode() == msg and msg != "no error"


def test_scatter_argument_checks(lib):
    v = ctypes.c_void_p
    f = lib.pa_reshape_and_cache
    assert f(v(16), v(16), 128, v(16), v(16), v(16), 0, 2, 64, 16, 8, 1, None) == 0   # no tokens
    assert f(v(16), v(16), 100, v(16), v(16), v(16), 4, 2, 64, 16, 8, 1, None) == 1   # stride < H*D
    assert f(None, v(16), 128, v(16), v(16), v(16), 4, 2, 64, 16, 8, 1, None) == 1    # null key
    assert f(v(16), v(16), 128, v(16), v(16), v(16), 4, 2, 64, 16, 8, 9, None) == 1   # dtype


def test_reduce_argument_checks(lib):
    v = ctypes.c_void_p
    f = lib.pa_split_kv_reduce
    assert f(v(16), v(16), v(16), v(16), v(16), v(16), 2, 4, 256, 4, 96, None, 1, None) == 2
    assert f(v(16), v(16), v(16), v(16), v(16), v(16), 2, 0, 256, 4, 64, None, 1, None) == 1
    assert f(None, v(16), v(16), v(16), v(16), v(16), 2, 4, 256, 4, 64, None, 1, None) == 1


def test_quantised_cache_argument_checks(lib):
    """The quantised-cache calls refuse what they do not take before any CUDA
    call: head_dim 64, float32 queries, missing scales, a bad dtype."""
    v = ctypes.c_void_p
    s = lib.pa_reshape_and_cache_fp8
    #        key    value   stride codes  codes  kscale vscale slots  T  Hkv D  bs nb dtype
    assert s(v(16), v(16), 256, v(16), v(16), v(16), v(16), v(16), 0, 2, 128, 16, 8, 1, None) == 0
    assert s(v(16), v(16), 128, v(16), v(16), v(16), v(16), v(16), 4, 2, 64, 16, 8, 1, None) == 2
    assert s(v(16), v(16), 128, v(16), v(16), v(16), v(16), v(16), 4, 2, 128, 16, 8, 1, None) == 1
    assert s(v(16), v(16), 256, v(16), v(16), None, v(16), v(16), 4, 2, 128, 16, 8, 1, None) == 1
    assert s(v(16), v(16), 256, v(16), v(16), v(16), v(16), v(16), 4, 2, 128, 16, 8, 9, None) == 1
    a = lib.pa_varlen_attention_fp8kv

    def call(D=128, dtype=1, ks=v(16)):
        return a(v(16), v(16), v(16), v(16), ks, v(16), v(16), v(16), v(16), 4, 2, 3, 2, 40, 8,
                 2, D, 16, 8, 0.1, None, 1, 0, None, 0, dtype, None)
    assert call(D=64) == 2                 # head_dim
    assert call(dtype=0) == 2              # float32 queries
    assert call(ks=None) == 1              # missing scales
    assert "scales" in lib.pa_last_error_string().decode()
