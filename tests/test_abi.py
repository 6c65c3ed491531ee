"""The C-ABI library builds, loads and exports every function include/moe.h declares, and
its host-side argument validation rejects bad calls before anything reaches a GPU.
(CPU only: no call here launches a kernel.)"""
import ctypes
import os
import re

import pytest

from expert_routed_ffn_router_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ctypes.CDLL(_build.LIB)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("moe_router_topk", "moe_dispatch", "moe_expert_ffn", "moe_combine",
              "moe_layer_forward", "moe_workspace_bytes", "moe_error_string",
              "moe_read_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_error_strings_and_workspace_size():
    assert binding.moe_error_string(0) == "ok"
    assert "timeout" in binding.moe_error_string(-6) or "ran out" in binding.moe_error_string(-6)
    n = binding.moe_workspace_bytes(128, 7168, 256, 8, 2048, 2048)
    # at least the permuted activations, h, Yp (bf16) and the shared output (fp32)
    TK = 128 * 8
    assert n >= TK * 7168 * 2 * 2 + TK * 2048 * 2 + 128 * 7168 * 4
    assert binding.moe_workspace_bytes(1, 100, 16, 2, 128, 0) == 0        # H % 64 != 0
    assert binding.moe_workspace_bytes(1, 256, 2048, 2, 128, 0) == 0      # E > 1024
    assert binding.moe_workspace_bytes(1, 256, 16, 17, 128, 0) == 0       # K > E
    assert binding.moe_workspace_bytes(0, 256, 16, 2, 128, 128) > 0


def test_validation_rejects_before_launch(lib):
    lib.moe_router_topk.restype = ctypes.c_int
    lib.moe_combine.restype = ctypes.c_int
    P = ctypes.c_void_p
    ok = P(0x10000)            # never dereferenced: every call below fails validation
    bad = P(0x10001)
    ws = P(0x100000)
    f = lib.moe_router_topk
    f.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P,
                  ctypes.c_size_t, P]
    assert f(ok, ok, ok, 4, 256, 16, 17, ok, ok, ws, 1 << 20, None) == -1   # K > E
    assert f(ok, ok, ok, 4, 96, 16, 2, ok, ok, ws, 1 << 20, None) == -2     # H % 64
    assert f(bad, ok, ok, 4, 256, 16, 2, ok, ok, ws, 1 << 20, None) == -3   # misaligned
    assert f(None, ok, ok, 4, 256, 16, 2, ok, ok, ws, 1 << 20, None) == -1  # null
    assert f(ok, ok, ok, 4, 256, 16, 2, ok, ok, ws, 16, None) == -4         # small ws
    assert f(ok, ok, ok, -1, 256, 16, 2, ok, ok, ws, 1 << 20, None) == -1   # T < 0
    g = lib.moe_combine
    g.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    assert g(ok, ok, ok, bad, 4, 256, 2, ok, None) == -3                    # Ysh misaligned
    assert g(ok, ok, ok, None, 4, 256, 33, ok, None) == -2                  # K > 32
    assert g(ok, ok, ok, None, 0, 256, 2, ok, None) == 0                    # T == 0: no-op


def test_routing_options_are_validated_before_launch(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.moe_router_topk_ex
    f.restype = I
    f.argtypes = [P, P, P, I, I, I, I, ctypes.POINTER(binding.MoeRouting), P, P, P,
                  ctypes.c_size_t, P]
    ok = P(0x10000)            # never dereferenced: every call below fails validation
    ws = P(0x100000)

    def call(E, K, **kw):
        r = binding.MoeRouting.make(**kw)
        return f(ok, ok, ok, 4, 256, E, K, ctypes.byref(r), ok, ok, ws, 16, None)

    # options that define no selection -> MOE_ERR_INVALID_ARG
    assert call(16, 2, n_group=3) == -1                         # 3 does not divide 16
    assert call(16, 2, n_group=4, topk_group=5) == -1           # more groups kept than exist
    assert call(16, 2, n_group=4, topk_group=0) == -1
    assert call(16, 9, n_group=4, topk_group=2) == -1           # K > 2 groups x 4 experts
    assert call(16, 2, n_group=4, topk_group=2, group_top=5) == -1
    r = binding.MoeRouting(2, 1, 1, 1, 1)                       # scoring 2 is undefined
    assert f(ok, ok, ok, 4, 256, 16, 2, ctypes.byref(r), ok, ok, ws, 16, None) == -1
    # defined but outside the kernel's support -> MOE_ERR_UNSUPPORTED_SHAPE
    assert call(128, 2, n_group=64, topk_group=2) == -2
    assert call(16, 2, n_group=2, topk_group=1, group_top=3) == -2
    # valid options reach the next check (the 16-byte workspace is too small)
    assert call(16, 2, n_group=4, topk_group=2, group_top=2, scoring="softmax") == -4
    assert f(ok, ok, ok, 4, 256, 16, 2, None, ok, ok, ws, 16, None) == -4   # NULL = defaults


@pytest.mark.parametrize("shape", [(128, 7168, 256, 8, 2048, 2048), (16, 256, 16, 2, 128, 128),
                                   (1, 64, 1, 1, 64, 0), (16384, 7168, 256, 8, 2048, 2048)])
def test_workspace_layout_lies_inside_the_workspace(shape):
    T, H, E, K, I, Is = shape
    lay = binding.moe_workspace_layout(*shape)
    assert lay["bytes"] == binding.moe_workspace_bytes(*shape)
    ends = [("offsets", (E + 1) * 4), ("perm", T * K * 4), ("slot_pos", T * K * 4),
            ("Xp", T * K * H * 2), ("h", T * K * I * 2), ("Yp", T * K * H * 2)]
    prev_end = 256                      # the status header comes first
    for name, nbytes in ends:
        assert lay[name] % 256 == 0, name
        assert lay[name] >= prev_end, name
        prev_end = lay[name] + nbytes
    assert prev_end <= lay["bytes"]
    if Is:
        assert lay["Ysh"] % 256 == 0 and lay["Ysh"] + T * H * 4 <= lay["bytes"]


def test_workspace_layout_rejects_what_the_size_query_rejects():
    with pytest.raises(binding.MoeError):
        binding.moe_workspace_layout(1, 100, 16, 2, 128, 0)       # H % 64 != 0


def test_binding_checks_element_types_and_sizes_before_the_call():
    # the C ABI takes bare pointers: the binding rejects a tensor of another element type,
    # or one smaller than the sizes passed beside it (which a kernel would read past),
    # before anything is called (CPU tensors: the checks come before the device check)
    import torch
    T, H, E, K = 4, 64, 8, 2
    X = torch.zeros(T, H, dtype=torch.bfloat16)
    Wg = torch.zeros(E, H, dtype=torch.bfloat16)
    bias = torch.zeros(E, dtype=torch.float32)
    idx = torch.zeros(T, K, dtype=torch.int32)
    wt = torch.zeros(T, K, dtype=torch.float32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError, match="X: dtype"):
        binding.moe_router_topk(X.float(), Wg, bias, K, idx, wt, ws)
    with pytest.raises(ValueError, match="W_gate: 256 elements, expected 512"):
        binding.moe_router_topk(X, Wg[:, :32].contiguous(), bias, K, idx, wt, ws)
    with pytest.raises(ValueError, match="topk_idx: dtype"):
        binding.moe_router_topk(X, Wg, bias, K, idx.long(), wt, ws)
    with pytest.raises(ValueError, match="device tensors"):
        binding.moe_router_topk(X, Wg, bias, K, idx, wt, ws)
    # the layer: a routed weight with fewer experts than the shape says
    shape = binding.MoeShape(T, H, E, K, 64, 0)
    W = {"W_gate": Wg, "bias": bias, "W1": torch.zeros(E - 1, H, 64, dtype=torch.bfloat16),
         "W3": torch.zeros(E, H, 64, dtype=torch.bfloat16),
         "W2": torch.zeros(E, 64, H, dtype=torch.bfloat16)}
    with pytest.raises(ValueError, match="W1: "):
        binding.moe_layer_forward(shape, W, X, torch.zeros(T, H), idx, wt,
                                  torch.zeros(E, dtype=torch.int32), None, ws)


def test_binding_checks_the_dispatch_ffn_and_combine_arguments():
    import torch
    T, H, E, K, I = 4, 64, 8, 2, 64
    X = torch.zeros(T, H, dtype=torch.bfloat16)
    idx = torch.zeros(T, K, dtype=torch.int32)
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)
    ws = torch.zeros(1024, dtype=torch.uint8)
    Xp = torch.zeros(T * K, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="perm: dtype"):
        binding.moe_dispatch(X, idx, E, i32(E), i32(E + 1), torch.zeros(T * K, dtype=torch.int64),
                             i32(T * K), Xp, None, ws)
    with pytest.raises(ValueError, match="offsets: 8 elements, expected 9"):
        binding.moe_dispatch(X, idx, E, i32(E), i32(E), i32(T * K), i32(T * K), Xp, None, ws)
    W = torch.zeros(E, H, I, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="Yp: dtype"):
        binding.moe_expert_ffn(Xp, i32(E + 1), E, W, W, W.transpose(1, 2).contiguous(),
                               torch.zeros(T * K, H, dtype=torch.float16), ws)
    with pytest.raises(ValueError, match="W2: "):
        binding.moe_expert_ffn(Xp, i32(E + 1), E, W, W, W[:-1].contiguous(),
                               torch.zeros(T * K, H, dtype=torch.float32), ws)
    with pytest.raises(ValueError, match="slot_pos: dtype"):
        binding.moe_combine(Xp, torch.zeros(T, K, dtype=torch.int64),
                            torch.zeros(T, K), None, torch.zeros(T, H))
