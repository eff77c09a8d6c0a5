"""C ABI checks that need no GPU: the library loads, exports every declared symbol, and rejects bad
arguments on the host before any launch."""
import ctypes
import re
import os

import pytest

import kda_gated_delta_rule_gb300 as kda
from kda_gated_delta_rule_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kda.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding_list():
    assert declared_functions() == sorted(kda.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_sizes(lib):
    assert kda.kda_status_string(0) == "KDA_OK"
    assert kda.kda_status_string(3) == "KDA_ERR_WORKSPACE"
    assert kda.kda_version() >= 10000
    assert kda.kda_state_bytes_per_head(128, 128) == 64 * 1024
    assert lib.kda_prefill_args_bytes() == ctypes.sizeof(kda.PrefillArgs)
    # raw-input record: 1028 bytes per token and head at d = 128, bf16 k/v (256 + 256 + 512 + 4)
    b = kda.kda_replay_bytes(256, 8, 12, 128, 128, 1)
    assert b >= 256 * 8 * 12 * 1028 and b - 256 * 8 * 12 * 1028 < 4 * 256


def test_stated_size_formulas(lib):
    """The sizes the header states in closed form: the backward's workspace is n = (ceil(T/64) + N) x H
    records of 574720 bytes, n operand records of 148480 bytes (each part rounded up to 1024 bytes), N x P x H
    x 196608 bytes of segment maps and entry states with P = max(1, 152 // H), and N x H int32 flags (rounded
    up to 256 bytes); a CF-BI row cache is 16 rows x 420 fp32 per head at d = 128 and 0 elsewhere."""
    up = lambda x, m: -(-x // m) * m
    for T, N, H in ((8192, 1, 12), (300, 3, 2), (64, 1, 1), (65, 2, 4), (1000, 1, 100)):
        n = (-(-T // 64) + N) * H
        P = max(1, 152 // H)
        want = up(n * 574720, 1024) + up(n * 148480, 1024) + N * P * H * 196608 + up(4 * N * H, 256)
        assert kda.kda_backward_workspace_size(T, N, H) == want
    assert kda.kda_cfbi_cache_bytes_per_head(128, 128) == kda.CFBI_CHUNK * kda.CFBI_ROW_FLOATS * 4 == 26880
    assert kda.kda_cfbi_cache_bytes_per_head(64, 64) == 0
    assert lib.kda_backward_args_bytes() == ctypes.sizeof(kda.BackwardArgs)
    assert lib.kda_fused_decode_args_bytes() == ctypes.sizeof(kda.FusedDecodeArgs)


def test_host_validation_rejects_before_launch(lib):
    """Invalid arguments return an error code; nothing is launched (no GPU is needed to check this)."""
    null = None
    # unsupported head size
    assert lib.kda_decode_step(16, 16, 16, 16, 16, 4, 2, 48, 48, 1, 16, 8, 16, 16, 1, null, null) == 2
    # null pointer
    assert lib.kda_decode_step(null, 16, 16, 16, 16, 4, 2, 128, 128, 1, 16, 8, 16, 16, 1, null, null) == 1
    # misaligned pointer
    assert lib.kda_decode_step(18, 16, 16, 16, 16, 4, 2, 128, 128, 1, 16, 8, 16, 16, 1, null, null) == 1
    # bad dtype
    assert lib.kda_decode_step(16, 16, 16, 16, 16, 4, 2, 128, 128, 7, 16, 8, 16, 16, 1, null, null) == 1
    # replay buffer too small
    assert lib.kda_verify(16, 16, 16, 16, 16, 4, 8, 2, 128, 128, 1, 16, 8, 16, 16, 1, 16, 100, null, null,
                          null) == 3
    # empty batches are no-ops
    assert lib.kda_decode_step(null, null, null, null, null, 0, 2, 128, 128, 1, null, 0, null, null, 1, null,
                               null) == 0
    assert lib.kda_state_copy(null, 0, null, null, 0, null, 0, 16, null, null) == 0
    assert lib.kda_state_copy(16, 4, 16, 16, 4, 16, 1, 18, null, null) == 1  # state_elems not a multiple of 4


def test_prefill_validation(lib):
    a = kda.PrefillArgs()
    a.q = a.k = a.v = a.g = a.beta = a.out = 16
    a.cu_seqlens = a.pool = a.slot_ids = 16
    a.in_dtype, a.out_dtype = 1, 1
    a.T, a.H, a.dk, a.dv, a.N, a.max_seqlen, a.num_slots = 64, 2, 128, 128, 1, 64, 1
    a.dk = a.dv = 96
    assert lib.kda_prefill_varlen(ctypes.byref(a), None) == 2
    a.dk = a.dv = 128
    # segment length must be a positive multiple of 64, and the workspace must be large enough
    assert lib.kda_prefill_segmented(ctypes.byref(a), 100, None) == 1
    assert lib.kda_prefill_segmented(ctypes.byref(a), 64, None) == 3
    need = lib.kda_segmented_workspace_size(ctypes.byref(a), 64)
    # bf16, d = 128: chunk records (ceil(T/64) + N) * H * 148480, then frag [N][P][H][dk][dv+dk] and
    # entry [N][P][H][dk][dv] in fp32 with P = ceil(64/64) = 1
    records = (1 + 1) * 2 * 148480
    assert lib.kda_prefill_workspace_size(ctypes.byref(a)) == records
    assert need == records + 2 * 128 * 256 * 4 + 2 * 128 * 128 * 4
    a.in_dtype = 0  # fp32 inputs take the token-sequential path: no records
    assert lib.kda_prefill_workspace_size(ctypes.byref(a)) == 0
    assert lib.kda_segmented_workspace_size(ctypes.byref(a), 64) == 2 * 128 * 256 * 4 + 2 * 128 * 128 * 4
    a.in_dtype = 1
    a.workspace, a.workspace_bytes = 16, need - 1
    assert lib.kda_prefill_segmented(ctypes.byref(a), 64, None) == 3
    # the tensor-core varlen path needs its records too
    a.workspace, a.workspace_bytes = 0, 0
    assert lib.kda_prefill_varlen(ctypes.byref(a), None) == 3
    a.N = -1
    assert lib.kda_prefill_varlen(ctypes.byref(a), None) == 1


def test_library_fails_loudly_when_missing(tmp_path, monkeypatch):
    """Without the built library there is no fallback: loading raises."""
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "absent" / "libkda.so"))
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(RuntimeError):
        kda.load()


def test_slot_id_contract_check_on_the_host(lib):
    """kda_check_slot_ids (host arrays): distinct ids pass; a repeated id, or an id shared with the other set
    (a copy whose destination is also its source, a snapshot into a sequence's own slot), is rejected."""
    import numpy as np
    ok, bad = kda.KDA_OK, 1  # KDA_ERR_INVALID_ARG
    assert kda.kda_check_slot_ids(np.array([3, 0, 7, 1])) == ok
    assert kda.kda_check_slot_ids(np.array([], np.int32)) == ok
    assert kda.kda_check_slot_ids(np.array([3, 0, 7, 3])) == bad
    assert kda.kda_check_slot_ids(np.array([5, 6]), other_ids=np.array([1, 2, 3])) == ok
    assert kda.kda_check_slot_ids(np.array([5, 6]), other_ids=np.array([1, 6, 3])) == bad
    # out-of-range ids are the device's to flag (KDA_DEV_SLOT_OOB), not this check's
    assert kda.kda_check_slot_ids(np.array([-1, 10 ** 6])) == ok
    assert lib.kda_check_slot_ids(None, -1, None, 0) == bad


def test_debug_checks_switch(lib):
    was = kda.kda_debug_checks()
    try:
        kda.kda_set_debug_checks(True)
        assert kda.kda_debug_checks() is True
        kda.kda_set_debug_checks(False)
        assert kda.kda_debug_checks() is False
    finally:
        kda.kda_set_debug_checks(was)


def test_test_fault_hook_values(lib):
    assert lib.kda_set_test_fault(99) == 1  # unknown value: KDA_ERR_INVALID_ARG
    assert lib.kda_set_test_fault(kda.KDA_TEST_FAULT_STALL_RECORD_INPUTS) == 0
    assert lib.kda_set_test_fault(kda.KDA_TEST_FAULT_NONE) == 0
