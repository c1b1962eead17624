"""CPU tests of the C ABI boundary: the library loads without a GPU, exports
every declared entry point, and its host-side planner and measurement
arithmetic agree with the figures printed on the pages (tests/golden)."""
import ctypes
import json
import os
import re

import pytest

from latency_barrier_free_gb300 import build_ext, measure, rra

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_figures.json")))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_ext.build()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(rra_\w+)\s*\(", text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(rra.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(names) == sorted(rra.SYMBOLS)


def test_status_strings_and_version():
    for code in range(7):
        assert rra.status_string(code)
    assert rra.status_string(5) == "a device-side wait timed out"
    assert re.match(r"^\d+\.\d+\.\d+$", rra.version())


def test_layout_defaults_are_the_pages_scratch_sizes():
    cap1 = GOLDEN["scratch_oneshot_bytes"]["value"]
    cap2 = GOLDEN["scratch_twoshot_ll128_bytes"]["value"]
    for n in (2, 4, 8, 64):
        lay = rra.plan_layout(n, 512 << 20)
        # one-shot sentinel: 2 parities x N slots fill the 4 MiB cap exactly
        assert 2 * n * lay["os_chunk"] <= cap1 and 2 * n * lay["os_chunk"] > cap1 - 32 * n
        # LL: same region bytes, half the payload per step (2 x sizeof(T))
        assert lay["ll_chunk"] * GOLDEN["ll_bytes_per_payload_byte"]["value"] in (lay["os_chunk"], lay["os_chunk"] - 16)
        assert lay["ll_bytes"] == lay["os_bytes"]
        # two-shot: RS + AG, 2 parities, N slots each, within 64 MiB
        assert 4 * n * lay["ts_part"] <= cap2 and 4 * n * lay["ts_part"] > cap2 - 64 * n
        assert lay["la_bytes"] <= cap2 + 4096
        assert lay["window_stride"] % 65536 == 0
        assert lay["total_bytes"] == lay["ctrl_bytes"] + n * lay["window_stride"]


def test_layout_small_messages_are_not_capped():
    lay = rra.plan_layout(4, 1000)
    assert lay["os_chunk"] == 1008 and lay["ll_chunk"] == 1008
    assert lay["ts_part"] == 16 * 16  # ceil(63 vectors / 4) = 16 vectors
    assert lay["la_part"] == 16 * 16


def test_layout_rejects_bad_arguments():
    for args in ((1, 1024), (65, 1024), (4, 0)):
        with pytest.raises(rra.RraError) as e:
            rra.plan_layout(*args)
        assert e.value.status == rra.ERR_INVALID_ARG
    with pytest.raises(rra.RraError):
        rra.plan_layout(64, 1 << 20, 1024, 0)  # 1 KiB one-shot cap cannot hold 2 x 64 slots


def test_sol_floor_formula_reproduces_the_pages_number():
    # Sec. VI: L_SoL = 2 L_L2_RTT + L_remote_store.  With the pages' 0.306 us
    # L2 figure, the 1.404 us floor implies a 0.792 us remote store.
    rtt = GOLDEN["sol_l2_rtt_us"]["value"]
    floor = GOLDEN["sol_floor_128B_2gpu_us"]["value"]
    store = floor - 2 * rtt
    assert abs(store - 0.792) < 1e-9
    assert abs(measure.sol_floor_ns(rtt * 1000, store * 1000) - floor * 1000) < 1e-6


def test_bandwidth_arithmetic():
    assert measure.algorithmic_bytes(8, 1 << 20) == 16 << 20
    assert abs(measure.hbm_gbs(8, 1 << 20, 1e-3) - 16.777216) < 1e-9
    assert abs(measure.busbw_gbs(8, 1 << 20, 1e-3) - 1.048576 * 2 * 7 / 8) < 1e-9
    assert measure.median([3, 1, 2]) == 2 and measure.median([4, 1, 2, 3]) == 2.5


def test_create_without_gpu_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(rra.RraError) as e:
        rra.Comm(4, 4096)
    assert e.value.status == rra.ERR_CUDA


def test_auto_selection_by_size_and_ranks():
    # the paper picks one-shot for small and two-shot for larger messages at a
    # given rank count; the GB300 crossovers differ from its GB200 ones
    # up to 16 ranks (bulk-copy push): the one-shot while N^2 M <= 8 / 2 / 4 / 8 MiB
    # at N <= 2 / 4 / 8 / 16
    assert rra.select_algo(4, 128) == "oneshot_cluster"
    assert rra.select_algo(4, 128 << 10) == "oneshot_cluster"  # N^2 M = 2 MiB
    assert rra.select_algo(4, (128 << 10) + 16) == "twoshot_cluster"
    assert rra.select_algo(4, 1 << 20) == "twoshot_cluster"
    assert rra.select_algo(2, 2 << 20, "bf16") == "oneshot_cluster"  # N^2 M = 8 MiB
    assert rra.select_algo(2, (2 << 20) + 16, "bf16") == "twoshot_cluster"
    assert rra.select_algo(3, 224 << 10) == "oneshot_cluster"  # 1.97 MiB
    assert rra.select_algo(3, 256 << 10) == "twoshot_cluster"
    assert rra.select_algo(8, 64 << 10, "bf16") == "oneshot_cluster"  # 4 MiB
    assert rra.select_algo(8, (64 << 10) + 16, "bf16") == "twoshot_cluster"
    assert rra.select_algo(16, 32 << 10) == "oneshot_cluster"  # 8 MiB
    assert rra.select_algo(16, 64 << 10) == "twoshot_cluster"
    # above 16 ranks: 16-CTA clusters hosting several ranks each; with the
    # bulk-copy push the one-shot while 16 N M <= 16 MiB
    assert rra.select_algo(17, 1 << 10) == "oneshot_cluster"
    assert rra.select_algo(64, 16 << 10) == "oneshot_cluster"
    assert rra.select_algo(64, (16 << 10) + 16) == "twoshot_cluster"
    assert rra.select_algo(32, 32 << 10) == "oneshot_cluster"
    assert rra.select_algo(32, (32 << 10) + 16) == "twoshot_cluster"
    assert rra.select_algo(20, 48 << 10) == "oneshot_cluster"
    assert rra.select_algo(64, 64 << 10) == "twoshot_cluster"
    assert rra.select_algo(64, 1 << 20) == "twoshot_cluster"
    twoshot = ("twoshot_cluster", "twoshot_direct")
    for n in (2, 4, 8, 16, 17, 64):  # once two-shot, always two-shot as the message grows
        picks = [rra.select_algo(n, 1 << k) for k in range(4, 31)]
        first = min(i for i, p in enumerate(picks) if p in twoshot)
        assert all(p in twoshot for p in picks[first:])
    with pytest.raises(rra.RraError):
        rra.select_algo(1, 128)


def _declarations():
    """name -> list of parameter declarations, from include/*.h."""
    out = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\**\s+\**(rra_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M):
            params = [p.strip() for p in m.group(2).split(",")]
            out[m.group(1)] = [] if params == ["void"] or params == [""] else params
    return out


def _kind(param):
    """Coarse C kind of one parameter declaration."""
    if "*" in param or "[" in param or param.split()[0] in ("rra_comm_t", "rra_stream_t"):
        return "pointer"
    base = param.replace("const ", "").split()[0]
    # size_t and uint64_t are the same 64-bit unsigned type on the 64-bit targets (as in ctypes)
    return {"size_t": "u64", "int": "int", "double": "double", "int64_t": "int64", "uint64_t": "u64",
            "rra_dtype_t": "int", "rra_algo_t": "int", "rra_attr_t": "int", "rra_status_t": "int"}.get(base, base)


def _ctype_kind(t):
    if t in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "pointer"
    return {ctypes.c_size_t: "u64", ctypes.c_uint64: "u64", ctypes.c_int: "int", ctypes.c_double: "double",
            ctypes.c_int64: "int64"}.get(t, repr(t))


def test_binding_prototypes_match_the_headers():
    """Every function the ctypes binding gives a prototype takes as many
    arguments, of the same coarse kinds, as its declaration in include/*.h."""
    decls = _declarations()
    lib = rra.load()
    checked = 0
    for name in rra.SYMBOLS:
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert name in decls, name
        want = [_kind(p) for p in decls[name]]
        got = [_ctype_kind(t) for t in fn.argtypes]
        assert got == want, (name, got, want)
        checked += 1
    assert checked >= 30
