"""The C ABI library loads and exports every symbol include/river.h declares
(no compute calls: runs without a GPU)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "river.h")).read()
    return sorted(set(re.findall(r"^RL_API [^(]*?\b(rl_\w+)\(", src, flags=re.M)))


def test_header_declares_the_method_calls():
    names = _declared()
    for required in ("rl_quantize_exit_layers", "rl_prefill", "rl_decode_step", "rl_kv_cache_alloc"):
        assert required in names
    assert len(names) >= 17


def test_library_builds_and_exports_every_declared_symbol():
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_gb300 as river
    lib = ctypes.CDLL(river.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), f"libriver.so does not export {n}"
    assert set(_declared()) == set(river.EXPORTS)


def test_host_side_argument_errors_need_no_gpu():
    import early_exit_decoding_gb300 as river
    import pytest
    with pytest.raises(river.RiverError) as e:
        river.rl_kv_cache_alloc(None, 1, 16)
    assert e.value.status == river.RL_ERR_INVALID_ARG
    assert river.rl_decode_kernel_count(None, 1) == 0
    assert "NULL" in river.rl_last_error() or river.rl_last_error()


def test_failure_injection_hooks_are_host_side():
    """The allocation-failure hook is a host-side switch: it can be set and
    cleared without a GPU, and rl_kv_set_wait_limit rejects a NULL cache."""
    import early_exit_decoding_gb300 as river
    import pytest
    river.rl_debug_fail_allocations(3)
    river.rl_debug_fail_allocations(-1)
    with pytest.raises(river.RiverError) as e:
        river.rl_kv_set_wait_limit(None, 1)
    assert e.value.status == river.RL_ERR_INVALID_ARG
