"""Guard regions around every buffer the library writes (the padded-lane write
class the MI300X post reports: a write past a buffer's end under load).

Each output and the workspace sit inside a larger allocation whose head and
tail are filled with a byte pattern; after the call through the C ABI the
pattern must be intact, the inputs unchanged, and the results identical to
an ordinary call.  Kept last in the suite (file name) because it allocates
its own buffers around the library's.
"""
import ctypes

import numpy as np
import pytest

from moe_inputs import make_layer

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes before and after each buffer (keeps 256-byte alignment)
PATTERN = 0xA5
GEMV, TC, DET = 0x1, 0x2, 0x10


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import fp4_mixture_experts_gb300 as m
    m.load_library()
    return m


class Guarded:
    """nbytes of writable space with PATTERN-filled guards on both sides."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + GUARD)

    def view(self, dtype, shape):
        return self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == PATTERN).all() and (b[GUARD + self.nbytes:] == PATTERN).all())


def stream_ptr():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def device_inputs(L):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dict(x=t(L.x_bf16.view(np.int16)).view(torch.bfloat16), logits=t(L.router_logits), w13=t(L.w13),
                w13s=t(L.w13_scale), w2=t(L.w2), w2s=t(L.w2_scale))


@pytest.mark.parametrize("shape,flags", [((32, 1024, 1024, 64, 8), GEMV), ((70, 384, 640, 12, 3), TC),
                                         ((40, 1024, 1024, 16, 4), 0), ((32, 1024, 1024, 64, 8), GEMV | DET),
                                         ((70, 384, 640, 12, 3), TC | DET)])
def test_forward_writes_only_inside_its_buffers(moe, shape, flags):
    T, d, I, E, k = shape
    L = make_layer(T=T, d=d, I=I, E=E, k=k, seed=61 + T)
    D = device_inputs(L)
    before = {n: v.clone() for n, v in D.items()}
    lib = moe.load_library()
    dims = moe.Dims(T, d, I, E, k)
    S = T * k
    ws_bytes = moe.workspace_bytes(T, d, I, E, k)
    g = dict(out=Guarded(T * d * 4), ids=Guarded(S * 4), w=Guarded(S * 4), off=Guarded((E + 1) * 4),
             ss=Guarded(S * 4), h=Guarded(S * I * 2), ws=Guarded(ws_bytes))
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.moe_fp4_forward(ctypes.byref(dims), P(D["x"]), P(D["logits"]), P(D["w13"]), P(D["w13s"]), P(D["w2"]),
                             P(D["w2s"]), g["out"].ptr, g["ids"].ptr, g["w"].ptr, g["off"].ptr, g["ss"].ptr,
                             g["h"].ptr, flags, g["ws"].ptr, ws_bytes, stream_ptr())
    assert rc == 0
    torch.cuda.synchronize()
    for name, buf in g.items():
        assert buf.intact(), f"write outside {name}"
    for name, v in D.items():
        assert torch.equal(v, before[name]), f"input {name} changed"
    ref = moe.forward(D["x"], D["logits"], D["w13"], D["w13s"], D["w2"], D["w2s"], k, flags=flags,
                      return_routing=True, return_h=True)
    torch.cuda.synchronize()
    if flags & DET:
        assert torch.equal(g["out"].view(torch.float32, (T, d)), ref["out"])
    else:
        # the epilogue combine adds the k terms (the streaming kernel: 2k half-K
        # terms) in no fixed order: equal up to fp32 rounding of the partial sums
        x = g["out"].view(torch.float32, (T, d)).cpu().double().numpy()
        y = ref["out"].cpu().double().numpy()
        scale = np.abs(y).max(axis=1, keepdims=True)
        assert (np.abs(x - y) <= 4 * k * k * 2.0 ** -24 * scale).all()
    assert torch.equal(g["ids"].view(torch.int32, (T, k)), ref["topk_ids"])
    assert torch.equal(g["w"].view(torch.float32, (T, k)), ref["topk_weights"])
    assert torch.equal(g["off"].view(torch.int32, (E + 1,)), ref["expert_offsets"])
    assert torch.equal(g["ss"].view(torch.int32, (S,)), ref["sorted_slot"])
    assert torch.equal(g["h"].view(torch.int16, (S, I)), ref["h"].view(torch.int16))


@pytest.mark.parametrize("T,E,k", [(32, 256, 8), (77, 64, 6)])
def test_route_writes_only_inside_its_buffers(moe, T, E, k):
    L = make_layer(T=T, d=128, I=128, E=E, k=k, seed=71 + T)
    logits = torch.from_numpy(L.router_logits).cuda()
    before = logits.clone()
    lib = moe.load_library()
    dims = moe.Dims(T, 128, 128, E, k)
    S = T * k
    ws_bytes = moe.workspace_bytes(T, 128, 128, E, k)
    g = dict(ids=Guarded(S * 4), w=Guarded(S * 4), off=Guarded((E + 1) * 4), ss=Guarded(S * 4),
             ws=Guarded(ws_bytes))
    rc = lib.moe_fp4_route(ctypes.byref(dims), ctypes.c_void_p(logits.data_ptr()), g["ids"].ptr, g["w"].ptr,
                           g["off"].ptr, g["ss"].ptr, g["ws"].ptr, ws_bytes, stream_ptr())
    assert rc == 0
    torch.cuda.synchronize()
    for name, buf in g.items():
        assert buf.intact(), f"write outside {name}"
    assert torch.equal(logits, before)
    ids, w, off, ss = moe.route(logits, k)
    torch.cuda.synchronize()
    assert torch.equal(g["ids"].view(torch.int32, (T, k)), ids)
    assert torch.equal(g["off"].view(torch.int32, (E + 1,)), off)
    assert torch.equal(g["ss"].view(torch.int32, (S,)), ss)


def test_mxfp8_quantize_writes_only_inside_its_buffers(moe):
    R, K = 33, 96                       # 3 scale bytes per row: an odd total
    L = make_layer(T=R, d=K, I=32, E=1, k=1, seed=81)
    x = torch.from_numpy(L.x_bf16.view(np.int16)).view(torch.bfloat16).cuda()
    g = dict(codes=Guarded(R * K), scales=Guarded(R * K // 32))
    rc = moe.load_library().moe_fp4_mxfp8_quantize(ctypes.c_void_p(x.data_ptr()), R, K, g["codes"].ptr,
                                                    g["scales"].ptr, stream_ptr())
    assert rc == 0
    torch.cuda.synchronize()
    for name, buf in g.items():
        assert buf.intact(), f"write outside {name}"
    codes, scales = moe.mxfp8_quantize(x)
    torch.cuda.synchronize()
    assert torch.equal(g["codes"].view(torch.uint8, (R, K)), codes)
    assert torch.equal(g["scales"].view(torch.uint8, (R, K // 32)), scales)
