"""Host-side checks of libmsda that need no GPU.

The library must build, load, export every entry point include/msda.h
declares, and reject invalid arguments on the host before any CUDA call (so
these run on a machine without a GPU). No compute call is made here.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def so():
    from scale_deformable_attention_msda_gb300 import binding, build
    build.build()
    return binding.load()


def _declared_symbols():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"MSDA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_header_declares_the_api():
    names = _declared_symbols()
    from scale_deformable_attention_msda_gb300.binding import EXPORTED
    for n in EXPORTED:
        assert n in names


def test_library_exports_every_declared_symbol(so):
    for name in _declared_symbols():
        assert hasattr(so, name), name


def test_library_exports_nothing_else(so):
    import subprocess
    from scale_deformable_attention_msda_gb300 import build
    for lib in (build.LIBRARY, build.CHECKED_LIBRARY):
        out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True,
                             text=True, check=True).stdout
        exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
        assert exported == set(_declared_symbols()), lib


def test_checked_build_flag(so):
    """libmsda.so is the plain build, libmsda_checked.so the range-checked one
    (the flag is a constant: no CUDA call)."""
    from scale_deformable_attention_msda_gb300 import binding, build
    assert so.msda_checked_build() == 0
    assert binding.load(build.CHECKED_LIBRARY).msda_checked_build() == 1


def test_status_strings_and_version(so):
    for s in range(8):
        assert so.msda_status_string(s)
    assert so.msda_status_string(99) == b"unknown status"
    assert so.msda_version() >= 100


def test_sample_split_setting(so):
    """-1..3 are accepted (no CUDA call); anything else is MSDA_ERR_SHAPE and
    leaves the setting alone."""
    for v in (0, 1, 2, 3, -1):
        assert so.msda_set_sample_split(v) == 0
    for v in (-2, 4, 99):
        assert so.msda_set_sample_split(v) == 2
    assert so.msda_set_sample_split(-1) == 0


def _dims(**kw):
    from scale_deformable_attention_msda_gb300.binding import msda_dims_t
    d = dict(B=2, S=22223, Q=300, M=8, D=32, L=4, K=4)
    d.update(kw)
    return msda_dims_t(**d)


FAKE = 0x10000   # 16-byte aligned address; every call below fails validation or is
                 # empty, so no kernel is ever launched with it


def _fwd(so, dims, dtype=0, value=FAKE, shapes=FAKE, starts=FAKE, loc=FAKE, attn=FAKE,
         out=FAKE, order=None):
    vp = ctypes.c_void_p
    return so.msda_forward(vp(value), vp(shapes), vp(starts), vp(loc), vp(attn), vp(order),
                           vp(out), ctypes.byref(dims) if dims is not None else None, dtype,
                           vp(0))


def _bwd(so, dims, dtype=0, accum=1, ws=FAKE, ws_bytes=1 << 40, grad_value=FAKE, **kw):
    vp = ctypes.c_void_p
    return so.msda_backward(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(None),
                            vp(FAKE), vp(grad_value), vp(FAKE), vp(FAKE), vp(ws),
                            ctypes.c_size_t(ws_bytes), accum, ctypes.byref(dims), dtype, vp(0))


def test_validation_errors_before_any_launch(so):
    assert _fwd(so, None) == 1                                   # NULL dims
    assert _fwd(so, _dims(), dtype=7) == 3                       # bad dtype
    assert _fwd(so, _dims(L=17)) == 2                            # too many levels
    assert _fwd(so, _dims(L=0)) == 2
    assert _fwd(so, _dims(K=0)) == 2
    assert _fwd(so, _dims(D=12)) == 2                            # not a power-of-two multiple of 4
    assert _fwd(so, _dims(D=256)) == 2                           # fp32: D/4 = 64 lanes > 32
    assert _fwd(so, _dims(S=0)) == 2
    assert _fwd(so, _dims(B=-1)) == 2
    assert _fwd(so, _dims(S=2 ** 23, M=8, D=32)) == 2            # S*M*D >= 2^31
    assert _fwd(so, _dims(), value=None) == 1
    assert _fwd(so, _dims(), loc=None) == 1
    assert _fwd(so, _dims(), out=None) == 1
    assert _fwd(so, _dims(), value=FAKE + 4) == 4                # value not 16-byte aligned
    assert _fwd(so, _dims(), out=FAKE + 8) == 4
    assert _fwd(so, _dims(), loc=FAKE + 4) == 4                  # fp32 loc pairs need 8 bytes
    # bf16 pairs need only 4-byte alignment: the call gets past that check and
    # stops at the missing output (no call here reaches a launch)
    assert _fwd(so, _dims(), dtype=1, loc=FAKE + 4, out=None) == 1
    assert _fwd(so, _dims(), shapes=FAKE + 4) == 4
    assert _fwd(so, _dims(), order=FAKE + 2) == 4


def test_softmax_variant_size_limit(so):
    vp = ctypes.c_void_p
    # bf16, D = 32: 4 lanes per query-head, so at most 64 samples per query-head
    ok = _dims(L=4, K=16, Q=0)            # 64 samples, empty: valid, launches nothing
    big = _dims(L=4, K=17)                # 68 samples: refused before any launch
    args = lambda d: (vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(None), vp(FAKE),
                      ctypes.byref(d), 1, vp(0))
    assert so.msda_forward_softmax(*args(ok)) == 0
    assert so.msda_forward_softmax(*args(big)) == 2


def test_empty_problems_are_valid_and_launch_nothing(so):
    assert _fwd(so, _dims(B=0)) == 0
    assert _fwd(so, _dims(Q=0)) == 0
    assert _fwd(so, _dims(B=0), value=None, loc=None, attn=None, out=None) == 0
    assert _bwd(so, _dims(B=0)) == 0


def test_backward_workspace_rules(so):
    d = _dims()
    n = 2 * 22223 * 8 * 32
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 1, 1) == 4 * n     # bf16, fp32 buffer
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 2, 1) == 4 * n     # f16, fp32 buffer
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 1, 0) == 0         # native
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 0, 1) == 0         # fp32 data
    assert so.msda_backward_workspace_bytes(ctypes.byref(_dims(L=0)), 1, 1) == 0
    assert _bwd(so, d, dtype=1, accum=1, ws=None) == 5
    assert _bwd(so, d, dtype=1, accum=1, ws_bytes=4 * n - 1) == 5
    assert _bwd(so, d, dtype=1, accum=1, ws=FAKE + 8, ws_bytes=4 * n) == 4
    assert _bwd(so, d, dtype=1, accum=5) == 3
    assert _bwd(so, d, grad_value=None) == 1


def test_value_sized_byte_counts_cannot_wrap(so):
    """B*S*M*D is bounded (<= 2^60 elements) so that the fp32 workspace's byte
    count, B*S*M*D*4, can never wrap around: with S*M*D just under 2^31 and a
    huge B the dims are refused, and the workspace size is 0 (invalid), not a
    wrapped small number that would pass the size checks."""
    smd = 2 ** 31 - 2 ** 13                     # S*M*D < 2^31: allowed on its own
    d = _dims(S=smd // (8 * 32), M=8, D=32, B=2 ** 31 - 1, Q=1)
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 1, 1) == 0
    assert _bwd(so, d, dtype=1, accum=1) == 2
    assert _fwd(so, d) == 2
    static = so.msda_backward_static_workspace
    vp = ctypes.c_void_p
    assert static(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), vp(None), vp(FAKE), vp(FAKE),
                  vp(FAKE), vp(FAKE), ctypes.byref(d), 1, vp(0)) != 0
    ok = _dims(B=2 ** 20, Q=0)                  # large but B*S*M*D < 2^60: still valid
    assert so.msda_backward_workspace_bytes(ctypes.byref(ok), 1, 1) == 4 * 2 ** 20 * 22223 * 256


def test_auto_accumulation_is_resolved_from_the_sizes(so):
    """MSDA_ACC_AUTO is native when 4 Q K L <= 4 S (at most 4 corner adds per
    value row and head on average) and the fp32 buffer otherwise; the
    workspace size and every backward call agree (no CUDA call here)."""
    vp = ctypes.c_void_p
    dec = _dims(Q=300)                                  # 0.9 adds per row: native
    enc = _dims(Q=22223)                                # 64 adds per row: fp32 buffer
    n = 2 * 22223 * 8 * 32
    assert so.msda_backward_workspace_bytes(ctypes.byref(dec), 1, 2) == 0
    assert so.msda_backward_workspace_bytes(ctypes.byref(enc), 1, 2) == 4 * n
    assert so.msda_backward_workspace_bytes(ctypes.byref(enc), 0, 2) == 0          # fp32 data
    edge = _dims(Q=22223, K=1, L=1)                     # exactly 4 adds per row: native
    assert so.msda_backward_workspace_bytes(ctypes.byref(edge), 1, 2) == 0
    over = _dims(Q=22224, K=1, L=1)
    assert so.msda_backward_workspace_bytes(ctypes.byref(over), 1, 2) == 4 * n
    assert _bwd(so, enc, dtype=1, accum=2, ws=None) == 5          # the fp32 buffer needs one
    assert _bwd(so, dec, dtype=1, accum=2, grad_value=None) == 1  # native: no workspace asked
    assert so.msda_backward_zero(vp(FAKE), vp(None), ctypes.c_size_t(0), 2, ctypes.byref(enc),
                                 1, vp(0)) == 5
    assert _bwd(so, enc, dtype=1, accum=4) == 3                   # unknown mode
    assert _bwd(so, _dims(B=0), dtype=1, accum=2) == 0            # empty: nothing launched


def test_fp16_buffer_accumulation_rules(so):
    """MSDA_ACC_FP16_BUFFER: bf16 data needs B*S*M*D*2 + 20480 bytes and is
    taken only by the one-call backward (its zero step reads grad_out); other
    dtypes accumulate natively and need nothing (no CUDA call here)."""
    vp = ctypes.c_void_p
    d = _dims()
    n = 2 * 22223 * 8 * 32
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 1, 3) == 2 * n + 20480
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 2, 3) == 0      # fp16 data
    assert so.msda_backward_workspace_bytes(ctypes.byref(d), 0, 3) == 0      # fp32 data
    assert so.msda_backward_zero(vp(FAKE), vp(FAKE), ctypes.c_size_t(2 * n + 20480), 3,
                                 ctypes.byref(d), 1, vp(0)) == 3
    assert so.msda_backward_finish(vp(FAKE), ctypes.c_size_t(2 * n + 20480), vp(FAKE), 3,
                                   ctypes.byref(d), 1, vp(0)) == 3
    assert _bwd(so, d, dtype=1, accum=3, ws=None) == 5
    assert _bwd(so, d, dtype=1, accum=3, ws_bytes=2 * n + 20479) == 5
    assert _bwd(so, _dims(B=0), dtype=1, accum=3) == 0


def test_binding_refuses_cpu_tensors(so):
    from scale_deformable_attention_msda_gb300 import binding
    v = torch.zeros(1, 80, 2, 8)
    loc = torch.zeros(1, 4, 2, 2, 2, 2)
    attn = torch.zeros(1, 4, 2, 2, 2)
    shapes = torch.tensor([[8, 8], [4, 4]])
    starts = torch.tensor([0, 64])
    with pytest.raises(ValueError, match="CUDA"):
        binding.msda_forward(v, shapes, starts, loc, attn)


def test_graft_entry_build():
    import __graft_entry__
    __graft_entry__.build()
