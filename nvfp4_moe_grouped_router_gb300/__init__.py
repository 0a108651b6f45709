"""Python binding of libnvfp4moe, the sm_103a NVFP4 mixture-of-experts layer.

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind the C ABI declared in include/nvfp4moe.h.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing or the device is not a GB300 (compute capability 10.3), calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4moe.so")

NVF_F32, NVF_BF16, NVF_F16 = 0, 1, 2
LAYOUT_ROWMAJOR, LAYOUT_TILED, LAYOUT_TILED_GROUPED = 0, 1, 2
TILE_BYTES = 18432   # one (128-row, 256-K) chunk: 16 KB swizzled codes + 2 KB scale atoms
STATUS = {0: "NVF_OK", 1: "NVF_ERR_INVALID_ARG", 2: "NVF_ERR_UNSUPPORTED_DEVICE", 3: "NVF_ERR_WORKSPACE",
          4: "NVF_ERR_CUDA", 5: "NVF_ERR_TIMEOUT", 6: "NVF_ERR_DEVICE_CHECK"}

# Every entry point declared in include/nvfp4moe.h, with its ctypes signature.
_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "nvf_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvf_last_error_message": (ctypes.c_char_p, []),
    "nvf_abi_version": (_I32, []),
    "nvf_device_status": (ctypes.c_int, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "nvf_selftest_bounded_wait": (ctypes.c_int, [ctypes.c_uint64, _P]),
    "nvf_w13_row_map": (ctypes.c_int, [_I32, ctypes.POINTER(_I32)]),
    "nvfp4_tiled_bytes": (_SZ, [_I64, _I32, _I32]),
    "nvfp4_global_scale": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P]),
    "nvfp4_quantize": (ctypes.c_int, [_P, _I32, _I64, _I32, _I64, _P, _P, _P, _I32, _P, _P, _P, _I32, _P]),
    "nvfp4_prepare_weights": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "moe_route_permute_workspace_size": (ctypes.c_int, [_I32, _I32, ctypes.POINTER(_SZ)]),
    "moe_route_permute": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                         _SZ, _P]),
    "nvfp4_grouped_gemm": (ctypes.c_int, [_P, _I64, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _I64, _P]),
    "nvfp4_moe_workspace_layout": (ctypes.c_int, [_I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "moe_route_permute_noalloc": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                                 _P]),
    "nvfp4_moe_forward": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _P, _SZ, _P,
                                         _P]),
    "nvf_router_gemm": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _I64, _P]),
    "nvf_moe_graph_create": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _I32,
                                            ctypes.POINTER(ctypes.c_void_p)]),
    "nvf_moe_graph_launch": (ctypes.c_int, [_P, _P]),
    "nvf_moe_graph_destroy": (ctypes.c_int, [_P]),
    "nvfp4_w4a16_grouped_gemm": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P,
                                                _I64, _P]),
    "nvfp4_moe_forward_gated": (ctypes.c_int, [_P, _P, _I32, _P, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _P, _SZ,
                                               _P]),
    "nvf_ep_row_bytes": (_SZ, [_I32]),
    "nvf_ep_receive_scratch_words": (_SZ, [_I32, _I32]),
    "nvf_ep_dispatch": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                       _P]),
    "nvf_ep_receive": (ctypes.c_int, [_P, _I64, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "nvfp4_moe_experts": (ctypes.c_int, [_P, _P, _I64, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "nvf_ep_return": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P]),
    "nvf_moe_combine": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _I32, _I32, _I32, _P, _P]),
}


class NvfError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class MoEWeightsC(ctypes.Structure):
    _fields_ = [("E", _I32), ("H", _I32), ("I", _I32), ("shared", _I32), ("w13", _P), ("gs_w13", _P),
                ("w2", _P), ("gs_w2", _P)]


class WorkspaceLayoutC(ctypes.Structure):
    _fields_ = [(n, _SZ) for n in ("topk_ids", "topk_w", "expert_offsets", "tile_offsets", "perm_to_src",
                                    "src_to_perm", "perm_token", "route_scratch", "tile_group", "a1", "a2", "y",
                                    "logits", "total")] + [("R", _I64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m nvfp4_moe_grouped_router_gb300.build`"
                              " (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise NvfError(status, lib().nvf_last_error_message().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return NVF_F32
    if t.dtype == torch.bfloat16:
        return NVF_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


# ----------------------------------------------------------------------------- small helpers
def selftest_bounded_wait(limit_ns: int):
    """Launch the failure-detection self-test (a wait that gives up after limit_ns)."""
    _check(lib().nvf_selftest_bounded_wait(int(limit_ns), _stream()))


def device_status():
    """(code, detail) of the current device's error word (synchronises the stream, then clears it)."""
    code, detail = _I32(0), _I32(0)
    st = lib().nvf_device_status(_stream(), ctypes.byref(code), ctypes.byref(detail))
    if st not in (0, 5, 6):   # a device-reported timeout or failed device check: returned as the code
        _check(st)
    return code.value, detail.value


def w13_row_map(I: int):
    m = (_I32 * (2 * I))()
    _check(lib().nvf_w13_row_map(I, m))
    return list(m)


def tiled_bytes(rows: int, G: int, K: int) -> int:
    """Bytes of a tiled operand (G = 0: TILED, G >= 1: TILED_GROUPED)."""
    return int(lib().nvfp4_tiled_bytes(rows, G, K))


# ----------------------------------------------------------------------------- entry points
def global_scale(x: torch.Tensor, groups: int = 1) -> torch.Tensor:
    """gs[g] = amax(x[g]) / 2688 for x viewed as [groups, n]."""
    _cuda(x, "x")
    gs = torch.empty(groups, dtype=torch.float32, device=x.device)
    _check(lib().nvfp4_global_scale(_ptr(x), _dtype_code(x), groups, x.numel() // groups, _ptr(gs), _stream()))
    return gs


def quantize(x: torch.Tensor, gscale: torch.Tensor, layout: int = LAYOUT_ROWMAJOR, gather=None, offsets=None,
             tile_offsets=None, rows=None, codes=None, scales=None, groups: int = 1):
    """NVFP4 quantization of the rows of a 2-D tensor x.

    ROWMAJOR: returns (codes [rows, K/2], scales [rows, K/16]); tiled layouts:
    returns (buffer, None).  TILED (weights): rows form `groups` equal groups,
    group g quantized with gscale[g]."""
    _cuda(x, "x")
    K = x.shape[1]
    rows = (gather.numel() if gather is not None else x.shape[0]) if rows is None else rows
    G = offsets.numel() - 1 if offsets is not None else groups
    if codes is None:
        if layout == LAYOUT_ROWMAJOR:
            codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=x.device)
        else:
            codes = torch.zeros(max(tiled_bytes(rows, G if layout == LAYOUT_TILED_GROUPED else 0, K), 16),
                                dtype=torch.uint8, device=x.device)
    if scales is None and layout == LAYOUT_ROWMAJOR:
        scales = torch.empty(max(rows * (K // 16), 16), dtype=torch.uint8, device=x.device)
    _check(lib().nvfp4_quantize(_ptr(x), _dtype_code(x), rows, K, x.stride(0), _ptr(gather), _ptr(offsets),
                                _ptr(tile_offsets), G, _ptr(gscale), _ptr(codes), _ptr(scales), layout, _stream()))
    return codes, scales


def route_permute(logits: torch.Tensor, k: int, bias=None, renormalize=True, shared=False):
    _cuda(logits, "logits")
    T, E = logits.shape
    dev = logits.device
    R = T * k + (T if shared else 0)
    Et = E + int(shared)
    out = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device=dev),
               topk_w=torch.empty(T, k, dtype=torch.float32, device=dev),
               expert_offsets=torch.empty(Et + 1, dtype=torch.int32, device=dev),
               tile_offsets=torch.empty(Et + 1, dtype=torch.int32, device=dev),
               perm_to_src=torch.empty(R, dtype=torch.int32, device=dev),
               src_to_perm=torch.empty(R, dtype=torch.int32, device=dev),
               perm_token=torch.empty(R, dtype=torch.int32, device=dev))
    nbytes = _SZ(0)
    _check(lib().moe_route_permute_workspace_size(T, E, ctypes.byref(nbytes)))
    ws = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
    o = out
    _check(lib().moe_route_permute(_ptr(logits), _ptr(bias), T, E, k, int(renormalize), int(shared),
                                   _ptr(o["topk_ids"]), _ptr(o["topk_w"]), _ptr(o["expert_offsets"]),
                                   _ptr(o["tile_offsets"]), _ptr(o["perm_to_src"]), _ptr(o["src_to_perm"]),
                                   _ptr(o["perm_token"]), _ptr(ws), nbytes.value, _stream()))
    return out


def grouped_gemm(A, a_rows: int, B, gs_a, gs_b, offsets, tile_offsets, N: int, K: int, out_dtype=torch.float32,
                 D=None):
    """D[row] = gs_a[g] gs_b[g] A[row] . B[g]^T for the rows of group g.

    A: TILED_GROUPED buffer (K columns, up to a_rows rows); B: TILED buffer of the
    [G*N, K] weights.  Rows of D outside the groups are left untouched."""
    G = offsets.numel() - 1
    if D is None:
        D = torch.zeros(max(a_rows, 1), N, dtype=out_dtype, device=A.device)
    code = NVF_F32 if D.dtype == torch.float32 else NVF_BF16
    _check(lib().nvfp4_grouped_gemm(_ptr(A), a_rows, _ptr(B), _ptr(gs_a), _ptr(gs_b), _ptr(offsets),
                                    _ptr(tile_offsets), G, N, K, code, _ptr(D), D.stride(0), _stream()))
    return D


def w4a16_grouped_gemm(A, B, gs_b, offsets, tile_offsets, N: int, K: int, out_dtype=torch.float32, D=None):
    """D[row] = gs_b[g] A[row] . dB[g]^T for the rows of group g: A fp16 or bf16
    [rows, K] (row-major, grouped by offsets; bf16 is rounded to fp16 by the
    kernel), B the TILED weights of the groups."""
    _cuda(A, "A")
    if A.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("A must be float16 or bfloat16")
    G = offsets.numel() - 1
    rows = A.shape[0]
    if D is None:
        D = torch.zeros(max(rows, 1), N, dtype=out_dtype, device=A.device)
    code = NVF_F32 if D.dtype == torch.float32 else NVF_BF16
    a_code = NVF_F16 if A.dtype == torch.float16 else NVF_BF16
    _check(lib().nvfp4_w4a16_grouped_gemm(_ptr(A), a_code, rows, A.stride(0), _ptr(B), _ptr(gs_b), _ptr(offsets),
                                          _ptr(tile_offsets), G, N, K, code, _ptr(D), D.stride(0), _stream()))
    return D


# ----------------------------------------------------------------------------- the layer
@dataclass
class MoEWeights:
    E: int
    H: int
    I: int
    shared: bool
    w13: torch.Tensor     # TILED [E'*2I, H], prepared row order (w13_row_map)
    gs_w13: torch.Tensor  # float [E']
    w2: torch.Tensor      # TILED [E'*H, I]
    gs_w2: torch.Tensor

    def c_struct(self) -> MoEWeightsC:
        return MoEWeightsC(self.E, self.H, self.I, int(self.shared), self.w13.data_ptr(), self.gs_w13.data_ptr(),
                           self.w2.data_ptr(), self.gs_w2.data_ptr())


def prepare_weights(E: int, H: int, I: int, shared: bool, expert_fp32, device="cuda", chunk: int = 16) -> MoEWeights:
    """Prepare expert weights on the device with nvfp4_prepare_weights.

    expert_fp32(e) -> (w13 [2I, H], w2 [H, I]) float32 tensors (gate rows first,
    then up rows).  Experts are staged `chunk` at a time into one FP32 buffer
    and handed to the library, which computes the per-expert global scales, the
    NVFP4 rows, the w13 row order and the TILED layout.
    """
    Et = E + int(shared)
    w13 = torch.zeros(tiled_bytes(Et * 2 * I, 0, H), dtype=torch.uint8, device=device)
    w2 = torch.zeros(tiled_bytes(Et * H, 0, I), dtype=torch.uint8, device=device)
    gs13 = torch.empty(Et, dtype=torch.float32, device=device)
    gs2 = torch.empty(Et, dtype=torch.float32, device=device)
    n = max(1, min(chunk, Et))
    s13 = torch.empty(n, 2 * I, H, dtype=torch.float32, device=device)
    s2 = torch.empty(n, H, I, dtype=torch.float32, device=device)
    for e0 in range(0, Et, n):
        m = min(n, Et - e0)
        for i in range(m):
            a, b = expert_fp32(e0 + i)
            s13[i].copy_(a)
            s2[i].copy_(b)
        _check(lib().nvfp4_prepare_weights(_ptr(s13), _ptr(s2), NVF_F32, e0, m, H, I, _ptr(w13), _ptr(gs13),
                                           _ptr(w2), _ptr(gs2), _stream()))
    return MoEWeights(E, H, I, shared, w13, gs13, w2, gs2)


def workspace_layout(T: int, E: int, H: int, I: int, k: int, shared: bool) -> dict:
    L = WorkspaceLayoutC()
    _check(lib().nvfp4_moe_workspace_layout(T, E, H, I, k, int(shared), ctypes.byref(L)))
    return {n: getattr(L, n) for n, _ in L._fields_}


def workspace(T: int, w: MoEWeights, k: int) -> torch.Tensor:
    n = workspace_layout(T, w.E, w.H, w.I, k, w.shared)["total"]
    return torch.empty(max(n, 256), dtype=torch.uint8, device=w.w13.device)


def moe_forward(w: MoEWeights, x, logits, k: int, gs_a1, gs_a2, bias=None, renormalize=True,
                out_dtype=torch.float32, out=None, h_dump=None, ws=None, stage_events=None, cw=None):
    """The whole layer: route, permute, quantize, gate_up GEMM + SiLU*up requant, down GEMM, combine."""
    _cuda(x, "x")
    _cuda(logits, "logits")
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, w.H, dtype=out_dtype, device=x.device)
    if ws is None:
        ws = workspace(T, w, k)
    cw = w.c_struct() if cw is None else cw
    ev = None
    if stage_events is not None:
        ev = (ctypes.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
    _check(lib().nvfp4_moe_forward(ctypes.byref(cw), _ptr(x), _ptr(logits), _ptr(bias), T, k, int(renormalize),
                                   _ptr(gs_a1), _ptr(gs_a2), NVF_F32 if out.dtype == torch.float32 else NVF_BF16,
                                   _ptr(out), _ptr(h_dump), _ptr(ws), ws.numel(), ev, _stream()))
    return out


class MoEGraph:
    """One step of the layer captured as a CUDA graph (nvf_moe_graph_create):
    host-to-device copies of `x` and `logits` from page-locked host tensors,
    the layer, and the copy of the result into the page-locked host tensor
    `out`, all replayed by launch().  Fill x / logits, launch(), and read out
    after synchronizing the stream."""

    def __init__(self, w: MoEWeights, T: int, k: int, gs_a1, gs_a2, bias=None, renormalize=True,
                 out_dtype=torch.bfloat16):
        # x and logits in one page-locked buffer, logits right behind x: one copy a step
        xb, lb = T * w.H * 2, T * w.E * 4
        self._inputs = torch.zeros(xb + lb, dtype=torch.uint8).pin_memory()
        self.x = self._inputs[:xb].view(torch.bfloat16).view(T, w.H)
        self.logits = self._inputs[xb:].view(torch.float32).view(T, w.E)
        self.out = torch.zeros(T, w.H, dtype=out_dtype).pin_memory()
        self._keep = (w, gs_a1, gs_a2, bias)        # device buffers the graph reads
        cw = w.c_struct()
        h = ctypes.c_void_p()
        _check(lib().nvf_moe_graph_create(ctypes.byref(cw), T, k, int(renormalize), _ptr(gs_a1), _ptr(gs_a2),
                                          _ptr(bias), _ptr(self.x), _ptr(self.logits), _ptr(self.out),
                                          NVF_F32 if out_dtype == torch.float32 else NVF_BF16, ctypes.byref(h)))
        self._h = h

    def launch(self):
        _check(lib().nvf_moe_graph_launch(self._h, _stream()))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value is not None:
            torch.cuda.synchronize()
            lib().nvf_moe_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def router_gemm(x, w_gate, logits=None):
    """Router gate: logits = x . w_gate^T (bf16 in, float32 out) on the tensor cores."""
    _cuda(x, "x")
    _cuda(w_gate, "w_gate")
    if x.dtype != torch.bfloat16 or w_gate.dtype != torch.bfloat16:
        raise TypeError("x and w_gate must be bfloat16")
    T, H = x.shape
    n = w_gate.shape[0]
    if logits is None:
        logits = torch.empty(T, n, dtype=torch.float32, device=x.device)
    _check(lib().nvf_router_gemm(_ptr(x), _ptr(w_gate), T, H, n, _ptr(logits), logits.stride(0), _stream()))
    return logits


def moe_forward_gated(w: MoEWeights, x, w_gate, k: int, gs_a1, gs_a2, shared_gate=False, bias=None,
                      renormalize=True, out_dtype=torch.float32, out=None, ws=None, cw=None):
    """The layer from the hidden states: router gate, then the layer; shared_gate
    scales the shared expert's output by sigmoid of the gate's last row."""
    _cuda(x, "x")
    _cuda(w_gate, "w_gate")
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, w.H, dtype=out_dtype, device=x.device)
    if ws is None:
        ws = workspace(T, w, k)
    cw = w.c_struct() if cw is None else cw
    _check(lib().nvfp4_moe_forward_gated(ctypes.byref(cw), _ptr(w_gate), int(shared_gate), _ptr(x), _ptr(bias), T, k,
                                         int(renormalize), _ptr(gs_a1), _ptr(gs_a2),
                                         NVF_F32 if out.dtype == torch.float32 else NVF_BF16, _ptr(out), _ptr(ws),
                                         ws.numel(), _stream()))
    return out


# ----------------------------------------------------------------------------- expert parallelism
# Rank r of G owns routed experts [r E/G, (r+1) E/G); a shared expert is
# replicated.  The device steps are the library's; the exchanges below are
# torch.distributed all-to-alls (NCCL between GPUs, gloo between CPU ranks).

def ep_row_bytes(H: int) -> int:
    return int(lib().nvf_ep_row_bytes(H))


def ep_dispatch(x, route: dict, E: int, k: int, shared: bool, G: int, rank: int, gs_a1):
    """Quantized send rows (ranks' segments back to back), send_counts [G, E/G+1]
    and src_to_send [R] from one rank's tokens and routing."""
    _cuda(x, "x")
    T, H = x.shape
    R = T * k + (T if shared else 0)
    dev = x.device
    send = torch.empty(max(R, 1), ep_row_bytes(H), dtype=torch.uint8, device=dev)
    counts = torch.empty(G, E // G + 1, dtype=torch.int32, device=dev)
    s2s = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
    _check(lib().nvf_ep_dispatch(_ptr(x), T, H, E, k, int(shared), G, rank, _ptr(route["expert_offsets"]),
                                 _ptr(route["perm_token"]), _ptr(route["perm_to_src"]), _ptr(gs_a1), _ptr(send),
                                 _ptr(counts), _ptr(s2s), _stream()))
    return send[:R], counts, s2s[:R]


def ep_receive(recv_rows, recv_counts, El: int, shared: bool, H: int, n_recv: int):
    """Group the arriving rows by local expert: A1 (TILED_GROUPED), local offsets,
    local tile offsets and recv_to_grp."""
    G = recv_counts.shape[0]
    dev = recv_counts.device
    Et = El + int(shared)
    a1 = torch.empty(max(tiled_bytes(n_recv, Et, H), 16), dtype=torch.uint8, device=dev)
    off = torch.empty(Et + 1, dtype=torch.int32, device=dev)
    toff = torch.empty(Et + 1, dtype=torch.int32, device=dev)
    r2g = torch.empty(max(n_recv, 1), dtype=torch.int32, device=dev)
    g2r = torch.empty(max(n_recv, 1), dtype=torch.int32, device=dev)
    scratch = torch.empty(int(lib().nvf_ep_receive_scratch_words(G, El)), dtype=torch.int32, device=dev)
    _check(lib().nvf_ep_receive(_ptr(recv_rows), n_recv, _ptr(recv_counts), G, El, int(shared), H, _ptr(a1), _ptr(off),
                                _ptr(toff), _ptr(r2g), _ptr(g2r), _ptr(scratch), _stream()))
    return dict(a1=a1, offsets=off, tile_offsets=toff, recv_to_grp=r2g[:n_recv], grp_to_recv=g2r[:n_recv], n=n_recv)


def moe_experts(w: MoEWeights, a1, a_rows: int, offsets, tile_offsets, gs_a1, gs_a2, out_dtype=torch.float32,
                y_rows=None):
    """Steps 4-6 on grouped rows: y [a_rows, H]; with y_rows, grouped row p is
    stored as y row y_rows[p]."""
    dev = a1.device
    y = torch.empty(max(a_rows, 1), w.H, dtype=out_dtype, device=dev)
    ws = torch.empty(max(tiled_bytes(a_rows, w.E + int(w.shared), w.I), 256), dtype=torch.uint8, device=dev)
    cw = w.c_struct()
    _check(lib().nvfp4_moe_experts(ctypes.byref(cw), _ptr(a1), a_rows, _ptr(offsets), _ptr(tile_offsets), _ptr(gs_a1),
                                   _ptr(gs_a2), NVF_F32 if out_dtype == torch.float32 else NVF_BF16, _ptr(y),
                                   _ptr(y_rows), _ptr(ws), ws.numel(), _stream()))
    return y[:a_rows]


def ep_return(y, recv_to_grp):
    """y rows back in received order."""
    n, H = y.shape
    out = torch.empty(max(n, 1), H, dtype=y.dtype, device=y.device)
    _check(lib().nvf_ep_return(_ptr(y), n, H, NVF_F32 if y.dtype == torch.float32 else NVF_BF16, _ptr(recv_to_grp),
                               _ptr(out), _stream()))
    return out[:n]


def moe_combine(y, topk_w, src_to_row, T: int, k: int, shared: bool):
    """out[t] = sum_j w[t,j] y[src_to_row[t*k+j]] (+ the shared row), FP32 sums."""
    H = y.shape[1]
    out = torch.empty(T, H, dtype=y.dtype, device=y.device)
    _check(lib().nvf_moe_combine(_ptr(y), H, NVF_F32 if y.dtype == torch.float32 else NVF_BF16, _ptr(topk_w),
                                 _ptr(src_to_row), T, k, int(shared), _ptr(out), _stream()))
    return out


def ep_exchange_counts(send_counts, group=None):
    """All-to-all of the per-destination count rows: recv_counts[s] = source s's
    send_counts row for this rank."""
    import torch.distributed as dist
    recv = torch.empty_like(send_counts)
    dist.all_to_all_single(recv, send_counts.contiguous(), group=group)
    return recv


def ep_exchange_rows(send, send_splits, recv_splits, group=None):
    """All-to-all of row buffers: send's first send_splits[0] rows go to rank 0,
    ...; returns the rows from every source back to back."""
    import torch.distributed as dist
    recv = torch.empty((sum(recv_splits),) + tuple(send.shape[1:]), dtype=send.dtype, device=send.device)
    dist.all_to_all_single(recv, send.contiguous(), list(recv_splits), list(send_splits), group=group)
    return recv


def ep_local_scales(gs, E: int, G: int, rank: int, shared: bool):
    """The local experts' entries of a per-expert vector [E + shared]."""
    El = E // G
    parts = [gs[rank * El:(rank + 1) * El]] + ([gs[E:E + 1]] if shared else [])
    return torch.cat(parts).contiguous()


def ep_forward(w_local: MoEWeights, x, logits, k: int, E: int, gs_a1, gs_a2, shared=False, renormalize=True,
               out_dtype=torch.float32, group=None):
    """The layer with expert parallelism on this rank: route over all E experts,
    dispatch, exchange, the local experts, return, exchange back, combine.
    w_local: this rank's E/G experts (and the shared one); gs_a1, gs_a2: the
    layer's per-expert scales [E + shared] (global ids)."""
    import torch.distributed as dist
    G, rank = dist.get_world_size(group), dist.get_rank(group)
    T, H = x.shape
    El = E // G
    route = route_permute(logits, k, renormalize=renormalize, shared=shared)
    send, send_counts, s2s = ep_dispatch(x, route, E, k, shared, G, rank, gs_a1)
    recv_counts = ep_exchange_counts(send_counts, group)
    # the split sizes are needed on the host (one small device-to-host copy)
    send_splits = send_counts.sum(dim=1).tolist()
    recv_splits = recv_counts.sum(dim=1).tolist()
    recv = ep_exchange_rows(send, send_splits, recv_splits, group)
    n_recv = sum(recv_splits)
    g = ep_receive(recv, recv_counts, El, shared, H, n_recv)
    # the down GEMM stores y rows in received order: the return exchange sends them as they are
    y_ret = moe_experts(w_local, g["a1"], n_recv, g["offsets"], g["tile_offsets"],
                        ep_local_scales(gs_a1, E, G, rank, shared), ep_local_scales(gs_a2, E, G, rank, shared),
                        out_dtype, y_rows=g["grp_to_recv"])
    y_back = ep_exchange_rows(y_ret, recv_splits, send_splits, group)
    return moe_combine(y_back, route["topk_w"], s2s, T, k, shared)
