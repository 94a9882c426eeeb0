"""Python binding of the FP8 linear-layer C ABI: torch allocates device buffers and supplies
the stream; every step of the computation runs in the library's CUDA kernels.

Names follow the C ABI: quantize, amax_update, linear_fwd, linear_bwd, gelu_quantize,
dgelu_quantize. A quantised tensor is a QTensor holding its torch buffers; its C view is
built on demand.
"""
import ctypes
from dataclasses import dataclass, field
from typing import Optional

import torch

from . import _lib as L

KINDS = {"delayed": L.RECIPE_DELAYED, "tensorwise": L.RECIPE_TENSORWISE,
         "mxfp8": L.RECIPE_MXFP8, "blockwise": L.RECIPE_BLOCKWISE}
ROLES = {"activation": L.ROLE_ACTIVATION, "weight": L.ROLE_WEIGHT, "grad": L.ROLE_GRAD}


@dataclass
class Recipe:
    """The recipe statement (--fp8-recipe, --fp8-format, --fp8-margin,
    --fp8-amax-history-len, --fp8-amax-compute-algo, --fp8-wgrad)."""
    kind: str = "delayed"
    format: str = "e4m3"
    margin: int = 0
    amax_history_len: int = 1024
    amax_compute_algo: str = "max"
    fp8_wgrad: bool = True
    power_2_scales: bool = False

    def c(self):
        return L.Recipe(KINDS[self.kind], 0 if self.format == "e4m3" else 1, int(self.margin),
                        int(self.amax_history_len), 0 if self.amax_compute_algo == "max" else 1,
                        1 if self.fp8_wgrad else 0, 1 if self.power_2_scales else 0)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class QTensor:
    """Codes and scales of one quantised tensor of source shape [rows, cols]."""
    rows: int
    cols: int
    kind: int
    role: int
    row: Optional[torch.Tensor] = None        # uint8 [rows, cols]
    col: Optional[torch.Tensor] = None        # uint8 [cols, rows]
    row_scale: Optional[torch.Tensor] = None
    col_scale: Optional[torch.Tensor] = None
    amax: Optional[torch.Tensor] = None       # float32 [1]
    scale: Optional[torch.Tensor] = None
    scale_inv: Optional[torch.Tensor] = None
    col_bf16: int = 0                         # 1: `col` is the bf16 transpose (wgrad in bf16)
    _c: object = field(default=None, repr=False)

    def c(self):
        t = L.Tensor()
        for name in ("row", "col", "row_scale", "col_scale", "amax", "scale", "scale_inv"):
            v = getattr(self, name)
            setattr(t, name, None if v is None else v.data_ptr())
        t.rows, t.cols, t.kind, t.role = self.rows, self.cols, self.kind, self.role
        t.col_bf16 = self.col_bf16
        self._c = t
        return t


def scale_shape(kind, role, rows, cols, pow2=False):
    """Storage of the scales of one copy whose codes are [rows, cols] (blocks along cols).
    Blockwise with power-of-two scales stores E8M0 bytes in the MXFP8 layout."""
    if kind == L.RECIPE_MXFP8 or (kind == L.RECIPE_BLOCKWISE and pow2):
        return (rows * cols // 32,), torch.uint8
    if kind == L.RECIPE_BLOCKWISE:
        if role == L.ROLE_WEIGHT:
            return (rows // 128, cols // 128), torch.float32
        return (cols // 128, rows), torch.float32
    return None, None


def empty_qtensor(recipe: Recipe, rows, cols, role="activation", want_row=True, want_col=True,
                  device="cuda"):
    kind, r = KINDS[recipe.kind], ROLES[role]
    q = QTensor(rows, cols, kind, r)
    if want_row:
        q.row = torch.empty((rows, cols), dtype=torch.uint8, device=device)
        shp, dt = scale_shape(kind, r, rows, cols, recipe.power_2_scales)
        if shp is not None:
            q.row_scale = torch.empty(shp, dtype=dt, device=device)
    if want_col:
        if not recipe.fp8_wgrad and r != L.ROLE_WEIGHT:
            # --fp8-wgrad off: the column copy is the bf16 transpose, read by the bf16 wgrad
            q.col = torch.empty((cols, rows), dtype=torch.bfloat16, device=device)
            q.col_bf16 = 1
        else:
            q.col = torch.empty((cols, rows), dtype=torch.uint8, device=device)
            shp, dt = scale_shape(kind, r, cols, rows, recipe.power_2_scales)
            if shp is not None:
                q.col_scale = torch.empty(shp, dtype=dt, device=device)
    if kind in (L.RECIPE_DELAYED, L.RECIPE_TENSORWISE):
        q.amax = torch.zeros(1, dtype=torch.float32, device=device)
        q.scale = torch.ones(1, dtype=torch.float32, device=device)
        q.scale_inv = torch.ones(1, dtype=torch.float32, device=device)
    return q


def workspace_bytes(recipe: Recipe, rows, cols):
    rc = recipe.c()
    return int(L.load().fp8_workspace_bytes(ctypes.byref(rc), rows, cols))


def quantize(recipe: Recipe, x: torch.Tensor, role="activation", want_row=True, want_col=True,
             out: Optional[QTensor] = None, workspace: Optional[torch.Tensor] = None,
             status: Optional[torch.Tensor] = None, stream=None):
    """fp8_quantize on a bf16 [rows, cols] tensor. For delayed scaling pass `out` whose
    scale / scale_inv hold the scale from the history (DelayedState.bind)."""
    lib = L.load()
    rows, cols = x.shape
    if out is None:
        out = empty_qtensor(recipe, rows, cols, role, want_row, want_col, device=x.device)
    rc = recipe.c()
    need = int(lib.fp8_workspace_bytes(ctypes.byref(rc), rows, cols))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ct = out.c()
    st = lib.fp8_quantize(ctypes.byref(rc), _ptr(x), rows, cols, ROLES[role], int(want_row),
                          int(want_col), ctypes.byref(ct), _ptr(workspace),
                          0 if workspace is None else workspace.numel(), _ptr(status),
                          _stream(stream))
    L.check(st, "fp8_quantize")
    out.rows, out.cols, out.kind, out.role = ct.rows, ct.cols, ct.kind, ct.role
    out.col_bf16 = ct.col_bf16
    return out


def quantize_group(recipe: Recipe, xs, roles, outs=None, want_row=True, want_col=True,
                   status: Optional[torch.Tensor] = None, stream=None, _stalled=False):
    """fp8_quantize_group: up to four bf16 [rows, cols] tensors quantised by one MXFP8 launch.
    `roles` and `outs` (QTensors, or None to allocate) run parallel to `xs`. `_stalled` calls
    the test hook fp8_test_quantize_group_stalled instead (the group's first tile never
    arrives, so CTA 0's bounded wait runs out and records FP8_ERR_TIMEOUT in `status`)."""
    lib = L.load()
    n = len(xs)
    if outs is None:
        outs = [None] * n
    outs = [o if o is not None else
            empty_qtensor(recipe, x.shape[0], x.shape[1], r, want_row, want_col, device=x.device)
            for x, r, o in zip(xs, roles, outs)]
    rc = recipe.c()
    cts = [o.c() for o in outs]
    items = (L.QuantizeItem * max(1, n))()
    for i, (x, r) in enumerate(zip(xs, roles)):
        items[i] = L.QuantizeItem(_ptr(x), x.shape[0], x.shape[1], ROLES[r], int(want_row),
                                  int(want_col), ctypes.pointer(cts[i]))
    fn = lib.fp8_test_quantize_group_stalled if _stalled else lib.fp8_quantize_group
    st = fn(ctypes.byref(rc), n, items, _ptr(status), _stream(stream))
    L.check(st, "fp8_quantize_group")
    for o, ct in zip(outs, cts):
        o.rows, o.cols, o.kind, o.role, o.col_bf16 = ct.rows, ct.cols, ct.kind, ct.role, ct.col_bf16
    return outs


def quantize_master(recipe: Recipe, w: torch.Tensor, want_row=True, want_col=True,
                    out: Optional[QTensor] = None, workspace: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None):
    """fp8_quantize_master on an fp32 [rows, cols] master weight (role weight, no bf16
    rounding). For delayed scaling pass `out` bound to the weight's DelayedState."""
    if w.dtype != torch.float32:
        raise TypeError("quantize_master takes fp32 master weights")
    lib = L.load()
    rows, cols = w.shape
    if out is None:
        out = empty_qtensor(recipe, rows, cols, "weight", want_row, want_col, device=w.device)
    rc = recipe.c()
    need = int(lib.fp8_workspace_bytes(ctypes.byref(rc), rows, cols))
    if need and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=w.device)
    ct = out.c()
    st = lib.fp8_quantize_master(ctypes.byref(rc), _ptr(w), rows, cols, int(want_row),
                                 int(want_col), ctypes.byref(ct), _ptr(workspace),
                                 0 if workspace is None else workspace.numel(), _ptr(status),
                                 _stream(stream))
    L.check(st, "fp8_quantize_master")
    out.rows, out.cols, out.kind, out.role = ct.rows, ct.cols, ct.kind, ct.role
    out.col_bf16 = ct.col_bf16
    return out


def quantize_static_scratch(recipe: Recipe, x: torch.Tensor, role="activation", want_row=True,
                            want_col=True, out: Optional[QTensor] = None, status=None,
                            stream=None):
    """fp8_quantize_static_scratch: like quantize(), but the library supplies the amax scratch
    from a fixed array in its device image, so the call allocates nothing (for callers that
    cannot allocate device memory). Calls that overlap on the GPU share that array and race."""
    lib = L.load()
    rows, cols = x.shape
    if out is None:
        out = empty_qtensor(recipe, rows, cols, role, want_row, want_col, device=x.device)
    rc = recipe.c()
    ct = out.c()
    st = lib.fp8_quantize_static_scratch(ctypes.byref(rc), _ptr(x), rows, cols, ROLES[role],
                                         int(want_row), int(want_col), ctypes.byref(ct),
                                         _ptr(status), _stream(stream))
    L.check(st, "fp8_quantize_static_scratch")
    out.rows, out.cols, out.kind, out.role = ct.rows, ct.cols, ct.kind, ct.role
    out.col_bf16 = ct.col_bf16
    return out


class DelayedState:
    """Device-resident delayed-scaling state: amax history, head, scale, scale_inv."""

    def __init__(self, recipe: Recipe, device="cuda", role="activation"):
        self.recipe = recipe
        self.role = role
        self.history = torch.zeros(recipe.amax_history_len, dtype=torch.float32, device=device)
        self.head = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = torch.ones(1, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(1, dtype=torch.float32, device=device)

    def bind(self, q: QTensor):
        """Point a QTensor's scale / scale_inv at this state (the cast reads them)."""
        q.scale, q.scale_inv = self.scale, self.scale_inv
        return q


def amax_update(recipe: Recipe, state: DelayedState, amax_new: torch.Tensor, stream=None):
    lib = L.load()
    rc = recipe.c()
    h = L.AmaxHistory(state.history.data_ptr(), state.head.data_ptr(), state.history.numel())
    st = lib.fp8_amax_update(ctypes.byref(rc), ctypes.byref(h), ROLES[state.role], _ptr(amax_new),
                             _ptr(state.scale), _ptr(state.scale_inv), _stream(stream))
    L.check(st, "fp8_amax_update")


def linear_fwd(recipe: Recipe, x: QTensor, w: QTensor, y: Optional[torch.Tensor] = None,
               fp32=False, status=None, stream=None):
    lib = L.load()
    if y is None:
        y = torch.empty((x.rows, w.rows), dtype=torch.float32 if fp32 else torch.bfloat16,
                        device=x.row.device)
    rc = recipe.c()
    st = lib.fp8_linear_fwd(ctypes.byref(rc), ctypes.byref(x.c()), ctypes.byref(w.c()), _ptr(y),
                            int(fp32), _ptr(status), _stream(stream))
    L.check(st, "fp8_linear_fwd")
    return y


def quantize_stalled(recipe: Recipe, x: torch.Tensor, role: str, out: QTensor,
                     status: torch.Tensor, stream=None):
    """Test hook (fp8_test_quantize_stalled): fp8_quantize with CTA 0's first tile never
    arriving, so its bounded wait runs out (about two seconds) and it records
    FP8_ERR_TIMEOUT in `status` (an int32 device word, zeroed by the caller)."""
    lib = L.load()
    rows, cols = x.shape
    rc = recipe.c()
    need = int(lib.fp8_workspace_bytes(ctypes.byref(rc), rows, cols))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    ct = out.c()
    st = lib.fp8_test_quantize_stalled(ctypes.byref(rc), _ptr(x), rows, cols, ROLES[role], 1, 1,
                                       ctypes.byref(ct), _ptr(ws), ws.numel(), _ptr(status),
                                       _stream(stream))
    L.check(st, "fp8_test_quantize_stalled")
    return out


def linear_fwd_stalled(recipe: Recipe, x: QTensor, w: QTensor, y: torch.Tensor,
                       status: torch.Tensor, stream=None):
    """Test hook (fp8_test_linear_fwd_stalled): fp8_linear_fwd with a pipeline stage that
    never becomes ready, so the kernel's bounded wait runs out (about two seconds) and it
    records FP8_ERR_TIMEOUT in `status` (an int32 device word, zeroed by the caller)."""
    lib = L.load()
    rc = recipe.c()
    st = lib.fp8_test_linear_fwd_stalled(ctypes.byref(rc), ctypes.byref(x.c()),
                                         ctypes.byref(w.c()), _ptr(y), _ptr(status),
                                         _stream(stream))
    L.check(st, "fp8_test_linear_fwd_stalled")
    return y


def linear_bwd(recipe: Recipe, dy: QTensor, x: Optional[QTensor], w: Optional[QTensor],
               want_dx=True, want_dw=True, dx=None, dw=None, fp32=False, status=None,
               stream=None):
    """dgrad (dy row copy x w column copy) and wgrad (dy and x column copies; bf16 when the
    recipe has fp8_wgrad off)."""
    lib = L.load()
    dt = torch.float32 if fp32 else torch.bfloat16
    dev = (dy.row if dy.row is not None else dy.col).device
    if want_dx and dx is None:
        dx = torch.empty((dy.rows, w.cols), dtype=dt, device=dev)
    if want_dw and dw is None:
        dw = torch.empty((dy.cols, x.cols), dtype=dt, device=dev)
    rc = recipe.c()
    cx = ctypes.byref(x.c()) if x is not None else None
    cw = ctypes.byref(w.c()) if w is not None else None
    st = lib.fp8_linear_bwd(ctypes.byref(rc), ctypes.byref(dy.c()), cx, cw,
                            _ptr(dx) if want_dx else None, _ptr(dw) if want_dw else None,
                            int(fp32), _ptr(status), _stream(stream))
    L.check(st, "fp8_linear_bwd")
    return dx, dw


def gelu_quantize(recipe: Recipe, h: torch.Tensor, want_a_bf16=False, a_q=None, h_q=None,
                  status=None, stream=None):
    """a = gelu(h) quantised (row + column copies) and h kept as an FP8 row copy."""
    lib = L.load()
    rows, cols = h.shape
    a_q = a_q or empty_qtensor(recipe, rows, cols, "activation", True, True, device=h.device)
    h_q = h_q or empty_qtensor(recipe, rows, cols, "activation", True, False, device=h.device)
    a_bf16 = torch.empty_like(h) if want_a_bf16 else None
    rc = recipe.c()
    ca, ch = a_q.c(), h_q.c()
    st = lib.fp8_gelu_quantize(ctypes.byref(rc), _ptr(h), rows, cols, _ptr(a_bf16),
                               ctypes.byref(ca), ctypes.byref(ch), _ptr(status), _stream(stream))
    L.check(st, "fp8_gelu_quantize")
    return a_q, h_q, a_bf16


def dgelu_quantize(recipe: Recipe, da: torch.Tensor, h_q: QTensor, want_dh_bf16=False,
                   dh_q=None, status=None, stream=None):
    """dh = da * gelu'(h) with h read from its FP8 copy, quantised (row + column copies)."""
    lib = L.load()
    rows, cols = da.shape
    dh_q = dh_q or empty_qtensor(recipe, rows, cols, "grad", True, True, device=da.device)
    dh_bf16 = torch.empty_like(da) if want_dh_bf16 else None
    rc = recipe.c()
    cd = dh_q.c()
    st = lib.fp8_dgelu_quantize(ctypes.byref(rc), _ptr(da), ctypes.byref(h_q.c()), _ptr(dh_bf16),
                                ctypes.byref(cd), _ptr(status), _stream(stream))
    L.check(st, "fp8_dgelu_quantize")
    return dh_q, dh_bf16


def linear_fwd_gelu(recipe: Recipe, x: QTensor, w: QTensor, a_q=None, h_q=None, status=None,
                    stream=None):
    """fc1 with GeLU fused into the GEMM epilogue: returns (a_q, h_q), the MXFP8 row and column
    copies of a = gelu(h) and the FP8 row copy of h = x . w^T; h is never stored in bf16."""
    lib = L.load()
    dev = x.row.device
    a_q = a_q or empty_qtensor(recipe, x.rows, w.rows, "activation", True, True, device=dev)
    h_q = h_q or empty_qtensor(recipe, x.rows, w.rows, "activation", True, False, device=dev)
    rc = recipe.c()
    st = lib.fp8_linear_fwd_gelu(ctypes.byref(rc), ctypes.byref(x.c()), ctypes.byref(w.c()),
                                 ctypes.byref(a_q.c()), ctypes.byref(h_q.c()), _ptr(status),
                                 _stream(stream))
    L.check(st, "fp8_linear_fwd_gelu")
    return a_q, h_q


def linear_dgrad_dgelu(recipe: Recipe, dy: QTensor, w: QTensor, h_q: QTensor, dh_q=None,
                       status=None, stream=None):
    """dgrad of fc2 with the GeLU backward fused: dh = (dy . w) * gelu'(h), h from its FP8 row
    copy, returned as MXFP8 row and column copies."""
    lib = L.load()
    dh_q = dh_q or empty_qtensor(recipe, dy.rows, w.cols, "grad", True, True,
                                 device=dy.row.device)
    rc = recipe.c()
    st = lib.fp8_linear_dgrad_dgelu(ctypes.byref(rc), ctypes.byref(dy.c()), ctypes.byref(w.c()),
                                    ctypes.byref(h_q.c()), ctypes.byref(dh_q.c()), _ptr(status),
                                    _stream(stream))
    L.check(st, "fp8_linear_dgrad_dgelu")
    return dh_q
