"""C ABI checks that need no GPU: the library builds, loads, exports every declared symbol,
and rejects bad arguments on the host before touching the device."""
import ctypes

import pytest

import block_draft_model_proj_gb300 as dflash
from block_draft_model_proj_gb300 import build as dbuild


@pytest.fixture(scope="module")
def cpu_lib():
    dbuild.build()
    return dflash.load()


def test_every_declared_symbol_is_exported(cpu_lib):
    names = dflash.declared_symbols()
    for required in ("dflash_plan", "dflash_project_context", "dflash_body_forward",
                     "dflash_verify_greedy", "dflash_last_error", "dflash_device_status"):
        assert required in names
    raw = ctypes.CDLL(dflash.LIB_PATH)
    missing = [n for n in names if not hasattr(raw, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(names) <= set(dflash._SIGS), set(names) - set(dflash._SIGS)


def test_version_and_error_string(cpu_lib):
    assert cpu_lib.dflash_version() >= 100
    assert isinstance(cpu_lib.dflash_last_error(), bytes)


def test_internal_symbols_are_hidden(cpu_lib):
    raw = ctypes.CDLL(dflash.LIB_PATH)
    assert not hasattr(raw, "_ZN6dflash10launch_gemm_tcEPKvlS2_lPfllliiPjP11CUstream_st")
    assert not hasattr(raw, "launch_plan")


def test_plan_rejects_bad_sizes_on_host(cpu_lib):
    st = cpu_lib.dflash_plan(None, None, 0, 10, 0, 0, 4, 16, None, None, None, None, None, None,
                             0, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    assert b"must be >= 1" in cpu_lib.dflash_last_error()
    st = cpu_lib.dflash_plan(None, None, 2, 10, 0, 0, 4, 16, None, None, None, None, None, None,
                             0, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    assert b"null" in cpu_lib.dflash_last_error()


def test_verify_rejects_bad_lengths_on_host(cpu_lib):
    # negative gamma: there is no way to have one target choice per draft token plus a bonus
    st = cpu_lib.dflash_verify_greedy(None, 1, None, 1, -1, 10, -1, None, None, None, None, None,
                                      0, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        dflash._check(st)


def test_config_validation_on_host(cpu_lib):
    import dflash_inputs as di
    cfg = dflash.make_config(di.QWEN3_8B_DRAFT)
    bad = dflash.make_config(di.QWEN3_8B_DRAFT)
    bad.num_kv_heads = 7
    w = dflash.dflash_weights_t()
    st = cpu_lib.dflash_body_forward(ctypes.byref(bad), ctypes.byref(w), None, None, None, None,
                                     None, None, 1, 1, 1, None, None, 0, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    assert b"multiple of num_kv_heads" in cpu_lib.dflash_last_error()
    st = cpu_lib.dflash_body_forward(ctypes.byref(cfg), None, None, None, None, None, None, None,
                                     1, 1, 1, None, None, 0, None)
    assert st == dflash.DFLASH_ERR_INVALID_ARG
    odd = dflash.make_config(di.QWEN3_8B_DRAFT)
    odd.hidden = 4100
    st = cpu_lib.dflash_body_forward(ctypes.byref(odd), ctypes.byref(w), None, None, None, None,
                                     None, None, 1, 1, 1, None, None, 0, None)
    assert st == dflash.DFLASH_ERR_UNSUPPORTED


def test_config_struct_layout_matches_header():
    assert ctypes.sizeof(dflash.dflash_config_t) == 12 * 4 + 2 * 8
    assert dflash.dflash_config_t.rope_theta.offset == 48
    assert ctypes.sizeof(dflash.dflash_layer_weights_t) == 6 * 8


@pytest.mark.parametrize("B,gamma,V", [(1, 15, 151936), (64, 15, 151936), (256, 15, 151936),
                                       (1024, 15, 151936), (1000, 15, 1001), (3, 0, 7),
                                       (16384, 0, 100000), (17, 962, 5003)])
@pytest.mark.parametrize("resident", [1, 152 * 8, 10 ** 6])
@pytest.mark.parametrize("entries", [0, 16384])
def test_verify_chunk_plan_covers_the_vocab(cpu_lib, B, gamma, V, resident, entries):
    """The argmax chunk plan (host arithmetic): chunks of a multiple of 8 elements that cover
    every vocab column exactly once; under the static variant's cap (16384 partials) the
    rows * chunks partials fit, even for a GPU with far more resident CTAs than this one."""
    rows = B * (gamma + 1)
    if entries and rows > entries:
        with pytest.raises(ValueError):
            dflash.dflash_testing_verify_plan(B, gamma, V, resident, entries)
        return
    chunks, clen = dflash.dflash_testing_verify_plan(B, gamma, V, resident, entries)
    assert clen % 8 == 0 and chunks >= 1
    assert chunks * clen >= V > (chunks - 1) * clen
    if entries:
        assert rows * chunks <= entries


def test_static_cap_branch_is_reached(cpu_lib):
    # with many resident CTAs the uncapped plan wants more partials than the static array
    # holds; the capped plan lengthens the chunks instead
    free = dflash.dflash_testing_verify_plan(1024, 15, 151936, 10 ** 6)
    capped = dflash.dflash_testing_verify_plan(1024, 15, 151936, 10 ** 6, 16384)
    assert free[0] * 1024 * 16 > 16384
    assert capped[0] == 1 and capped[1] >= 151936


def test_verify_rejects_gamma_beyond_the_scan_limit(cpu_lib):
    for fn in ("dflash_verify_greedy", "dflash_verify_greedy_static"):
        args = [None, 1, None, 1, 60000, 10, -1, None, None, None, None]
        if fn == "dflash_verify_greedy":
            args += [None, 0, None]
        else:
            args += [None]
        st = getattr(cpu_lib, fn)(*args)
        assert st == dflash.DFLASH_ERR_INVALID_ARG
        assert b"gamma" in cpu_lib.dflash_last_error()
