"""Host-side shape and dtype checks of the Python binding (no GPU needed).

Every entry point takes bare device pointers through the C ABI, so the binding checks each tensor against
the layout include/kda.h states before anything reaches the device.  A call whose tensors all match gets
past those checks and stops at the device check (these tensors live on the CPU); a call with one tensor of
the wrong shape or dtype raises an error that names that tensor.
"""
import pytest
import torch

import kda_gated_delta_rule_gb300 as kda

DEVICE_MSG = "expected contiguous CUDA tensors"
T, N, H, D, S, B, W = 70, 2, 2, 16, 5, 3, 4
BF, F32, I32 = torch.bfloat16, torch.float32, torch.int32


def z(*shape, dtype=F32):
    return torch.zeros(*shape, dtype=dtype)


def _prefill_kw():
    return dict(q=z(T, H, D, dtype=BF), k=z(T, H, D, dtype=BF), v=z(T, H, D, dtype=BF), g=z(T, H, D), beta=z(T, H),
                cu_seqlens=torch.tensor([0, 30, T], dtype=I32), max_seqlen=40, pool=z(S, H, D, D),
                slot_ids=z(N, dtype=I32), out=z(T, H, D))


def _decode_kw():
    return dict(q=z(B, H, D), k=z(B, H, D), v=z(B, H, D), g=z(B, H, D), beta=z(B, H), pool=z(S, H, D, D),
                slot_ids=z(B, dtype=I32), out=z(B, H, D, dtype=BF), dev_status=z(2, dtype=I32))


def _verify_kw():
    return dict(q=z(B, W, H, D, dtype=BF), k=z(B, W, H, D, dtype=BF), v=z(B, W, H, D, dtype=BF), g=z(B, W, H, D),
                beta=z(B, W, H), pool=z(S, H, D, D), slot_ids=z(B, dtype=I32), out=z(B, W, H, D),
                replay=z(64, dtype=torch.uint8), snapshot_out=z(B, W, H, D, D))


def _cfbi_state():
    return dict(pool=z(S, H, 128, 128), cache=z(S, H, kda.CFBI_CHUNK, kda.CFBI_ROW_FLOATS),
                counts=z(S, H, dtype=I32))


def _cfbi_prefill_kw():
    kw = _prefill_kw()
    for n in ("q", "k", "v", "g"):
        kw[n] = z(T, H, 128, dtype=kw[n].dtype)
    kw["out"] = z(T, H, 128)
    kw.update(_cfbi_state())
    return kw


def _cfbi_decode_kw():
    kw = dict(q=z(B, H, 128), k=z(B, H, 128), v=z(B, H, 128), g=z(B, H, 128), beta=z(B, H),
              slot_ids=z(B, dtype=I32), out=z(B, H, 128))
    kw.update(_cfbi_state())
    return kw


def _backward_kw():
    return dict(q=z(T, H, D), k=z(T, H, D), v=z(T, H, D), g=z(T, H, D), beta=z(T, H),
                cu_seqlens=torch.tensor([0, 30, T], dtype=I32), max_seqlen=40, d_out=z(T, H, D), dq=z(T, H, D),
                dk=z(T, H, D), dv=z(T, H, D), dg=z(T, H, D), dbeta=z(T, H), workspace=z(16, dtype=torch.uint8),
                pool=z(S, H, D, D), slot_ids=z(N, dtype=I32), d_final=z(N, H, D, D), d_init=z(N, H, D, D))


def _fused_kw():
    return dict(xq=z(B, H, 128, dtype=BF), xk=z(B, H, 128, dtype=BF), xv=z(B, H, 128, dtype=BF), a=z(B, H, 128),
                b=z(B, H), z=z(B, H, 128, dtype=BF), pool=z(S, H, 128, 128), slot_ids=z(B, dtype=I32),
                conv_state=z(S, H, 3, 3, 128), conv_w=z(3, H, 128, 4), norm_w=z(128), out=z(B, H, 128, dtype=BF))


def _copy_kw():
    return dict(src_pool=z(S, H, D, D), src_slots=z(B, dtype=I32), dst_pool=z(S + 2, H, D, D),
                dst_slots=z(B, dtype=I32))


def _replay_kw():
    return dict(pool=z(S, H, D, D), slot_ids=z(B, dtype=I32), replay=z(64, dtype=torch.uint8),
                accepted_len=z(B, dtype=I32), W=W, H=H, dk=D, dv=D, in_dtype=kda.BF16)


def _kcp_scan_kw():
    return dict(frags=z(3, H, D, 2 * D), s0=z(H, D, D), entries=z(3, H, D, D))


def _kcp_frag_kw():
    kw = _prefill_kw()
    kw.update(segment_len=64, workspace=z(16, dtype=torch.uint8), frag_out=z(N, 1, H, D, 2 * D))
    return kw


def _kcp_out_kw():
    kw = _prefill_kw()
    kw.update(segment_len=64, workspace=z(16, dtype=torch.uint8), entries=z(N, 1, H, D, D))
    return kw


def _segmented_kw():
    kw = _prefill_kw()
    kw.update(segment_len=64, workspace=z(16, dtype=torch.uint8))
    return kw


CALLS = {
    "kda_prefill_varlen": (kda.kda_prefill_varlen, _prefill_kw),
    "kda_prefill_segmented": (kda.kda_prefill_segmented, _segmented_kw),
    "kda_decode_step": (kda.kda_decode_step, _decode_kw),
    "kda_verify": (kda.kda_verify, _verify_kw),
    "kda_verify_replay": (kda.kda_verify_replay, _replay_kw),
    "kda_state_copy": (kda.kda_state_copy, _copy_kw),
    "kda_cfbi_prefill": (kda.kda_cfbi_prefill, _cfbi_prefill_kw),
    "kda_cfbi_decode": (kda.kda_cfbi_decode, _cfbi_decode_kw),
    "kda_prefill_backward": (kda.kda_prefill_backward, _backward_kw),
    "kda_fused_decode": (kda.kda_fused_decode, _fused_kw),
    "kda_kcp_fragments": (kda.kda_kcp_fragments, _kcp_frag_kw),
    "kda_kcp_scan": (kda.kda_kcp_scan, _kcp_scan_kw),
    "kda_kcp_outputs": (kda.kda_kcp_outputs, _kcp_out_kw),
}


def _bad_variants(kw):
    """(name, corrupted kwargs) for every tensor argument: one extent too many in its last dimension, an
    extra dimension, and a dtype the layout does not allow."""
    for name, t in kw.items():
        if not isinstance(t, torch.Tensor) or name in ("replay", "workspace"):
            continue  # byte buffers: any size, checked against the required bytes by the library
        if name == "dev_status":
            continue  # any int32 buffer of at least two elements (its own test below)
        grown = list(t.shape)
        grown[-1] += 1
        yield name, "shape", dict(kw, **{name: torch.zeros(*grown, dtype=t.dtype)})
        yield name, "rank", dict(kw, **{name: t.unsqueeze(0)})
        other = torch.float64 if t.dtype != torch.float64 else F32
        yield name, "dtype", dict(kw, **{name: t.to(other)})


@pytest.mark.parametrize("fn_name", sorted(CALLS))
def test_matching_tensors_reach_the_device_check(fn_name):
    fn, make = CALLS[fn_name]
    with pytest.raises(ValueError, match=DEVICE_MSG):
        fn(**make())


@pytest.mark.parametrize("fn_name", sorted(CALLS))
def test_each_mismatched_tensor_is_named(fn_name):
    fn, make = CALLS[fn_name]
    n = 0
    for name, kind, kw in _bad_variants(make()):
        with pytest.raises((ValueError, TypeError)) as e:
            fn(**kw)
        msg = str(e.value)
        assert DEVICE_MSG not in msg, f"{fn_name}: {kind} of {name} not caught on the host"
        # the message names an argument of the call: the corrupted tensor, or (when the corrupted one is the
        # tensor the others' extents are taken from) the first tensor that no longer matches it
        assert msg.split(":")[0] in kw, (fn_name, name, kind, msg)
        n += 1
    assert n > 0


def test_status_buffer_must_hold_two_int32():
    kw = _decode_kw()
    with pytest.raises(ValueError, match="dev_status"):
        kda.kda_decode_step(**dict(kw, dev_status=z(1, dtype=I32)))
    with pytest.raises(ValueError, match="dev_status"):
        kda.kda_decode_step(**dict(kw, dev_status=z(2, dtype=torch.int64)))


def test_paired_optional_arguments():
    kw = _prefill_kw()
    with pytest.raises(ValueError, match="extra_pool and extra_slot_ids"):
        kda.kda_prefill_varlen(**kw, extra_pool=z(4, H, D, D))
    bw = _backward_kw()
    with pytest.raises(ValueError, match="pool and slot_ids"):
        kda.kda_prefill_backward(**dict(bw, slot_ids=None))
