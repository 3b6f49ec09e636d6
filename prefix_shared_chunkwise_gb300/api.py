"""Thin Python binding over the C ABI: the same calls, with torch tensors for device
memory and streams.  Every step of the computation runs in the library's kernels;
this module only marshals pointers and sizes."""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib as L

__all__ = ["Plan", "kda_fwd", "kda_bwd", "conv_fwd", "conv_bwd", "semantic_map", "logprob_fwd",
           "logprob_bwd", "dtype_code"]


def dtype_code(torch_dtype):
    import torch
    if torch_dtype == torch.float32:
        return L.HARTS_FP32
    if torch_dtype == torch.bfloat16:
        return L.HARTS_BF16
    raise ValueError(f"unsupported dtype {torch_dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Plan:
    """harts_plan_calls + harts_plan_get_info / export / upload / free.

    nodewise=True asks for the node-wise plan (HARTS_PLAN_NODEWISE): one sequence per
    segment, one round per tree level.  noreplay=True asks for the no-replay plan
    (HARTS_PLAN_NOREPLAY, forward only): side branches start from the exact fork state."""

    def __init__(self, parent, seg_len, chunk: int, nodewise: bool = False, noreplay: bool = False):
        parent = np.ascontiguousarray(parent, np.int32)
        seg_len = np.ascontiguousarray(seg_len, np.int64)
        h = ctypes.c_void_p()
        flags = (L.HARTS_PLAN_NODEWISE if nodewise else 0) | (L.HARTS_PLAN_NOREPLAY if noreplay else 0)
        rc = L.lib().harts_plan_calls(len(parent), parent.ctypes.data_as(L._pi32),
                                      seg_len.ctypes.data_as(L._pi64), int(chunk), flags,
                                      ctypes.byref(h))
        L.check(rc, "harts_plan_calls")
        self._h = h
        info = L.PlanInfo()
        L.check(L.lib().harts_plan_get_info(self._h, ctypes.byref(info)), "harts_plan_get_info")
        self.info = {n: getattr(info, n) for n, _ in L.PlanInfo._fields_}
        self._dev = None

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            L.lib().harts_plan_free(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def arrays(self) -> dict:
        """Export every plan array into numpy (harts_plan_export)."""
        info = self.info
        env = dict(info)
        out, arr = {}, L.PlanArrays()
        for name, ty, size in L.PLAN_ARRAY_FIELDS:
            n = eval(size, {}, env)
            a = np.zeros(max(n, 1), np.int64 if ty == "i64" else np.int32)
            out[name] = (a, n)
            setattr(arr, name, a.ctypes.data_as(L._pi64 if ty == "i64" else L._pi32))
        L.check(L.lib().harts_plan_export(self._h, ctypes.byref(arr)), "harts_plan_export")
        return {k: a[:n] for k, (a, n) in out.items()}

    def device_bytes(self) -> int:
        return int(L.lib().harts_plan_device_bytes(self._h))

    def upload(self, device="cuda", stream=None):
        """Allocate the plan's device tables through torch and upload them."""
        import torch
        nb = self.device_bytes()
        buf = torch.empty(nb, dtype=torch.uint8, device=device)
        L.check(L.lib().harts_plan_upload(self._h, _ptr(buf), nb, _stream(stream)),
                "harts_plan_upload")
        self._dev = buf
        return self

    def device_error(self, stream=None) -> int:
        code = ctypes.c_int32(0)
        rc = L.lib().harts_plan_device_error(self._h, _stream(stream), ctypes.byref(code))
        if rc not in (0, -7):
            L.check(rc, "harts_plan_device_error")
        return code.value

    def chunk_state_bytes(self, H, dk, dv, dtype_c):
        return int(L.lib().harts_kda_chunk_state_bytes(self._h, H, dk, dv, dtype_c))

    def bwd_workspace_bytes(self, H, dk, dv):
        return int(L.lib().harts_kda_bwd_workspace_bytes(self._h, H, dk, dv))


def _need(name, t, shape=None, dtype=None, nbytes=None, device=None):
    """Size check of one buffer before its pointer crosses the C ABI (which cannot see sizes)."""
    if t is None:
        return
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, needs {nbytes}")


def _fwd_args(plan, q, k, v, g, beta, o, states, final_state, h0, chunk_states, scale, kernel):
    import torch
    C, H, dk = q.shape
    dv = v.shape[2]
    info, dev, f32 = plan.info, q.device, torch.float32
    if C != info["C"]:
        raise ValueError(f"q has {C} rows, the plan {info['C']}")
    for n, t, sh in (("k", k, (C, H, dk)), ("v", v, (C, H, dv)), ("g", g, (C, H, dk)),
                     ("beta", beta, (C, H)), ("o", o, (C, H, dv))):
        _need(n, t, sh, q.dtype, device=dev)
    per = H * dk * dv * 4                          # bytes of one fp32 state, all heads
    _need("states", states, None, f32, info["n_states"] * per, dev)
    _need("final_state", final_state, None, f32, info["n_seq"] * per, dev)
    _need("h0", h0, None, f32, info["n_roots"] * per, dev)
    _need("chunk_states", chunk_states, nbytes=plan.chunk_state_bytes(H, dk, dv, dtype_code(q.dtype)),
          device=dev)
    a = L.FwdArgs()
    a.H, a.dk, a.dv = H, dk, dv
    a.dtype = dtype_code(q.dtype)
    a.kernel = kernel
    a.scale = float(scale)
    for n, t in dict(q=q, k=k, v=v, g=g, beta=beta, o=o, states=states, final_state=final_state,
                     h0=h0, chunk_states=chunk_states).items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        setattr(a, n, None if t is None else t.data_ptr())
    return a


def kda_fwd(plan: Plan, q, k, v, g, beta, *, o=None, states=None, final_state=None, h0=None,
            chunk_states=None, scale=1.0, kernel=L.HARTS_KERNEL_AUTO, stream=None):
    """harts_kda_fwd.  Allocates any missing output through torch; returns
    (o, states, final_state, chunk_states)."""
    import torch
    C, H, dk = q.shape
    dv = v.shape[2]
    info = plan.info
    dev = q.device
    if o is None:
        o = torch.empty((C, H, dv), dtype=q.dtype, device=dev)
    if states is None and info["n_states"] > 0:
        states = torch.empty((info["n_states"], H, dk, dv), dtype=torch.float32, device=dev)
    a = _fwd_args(plan, q, k, v, g, beta, o, states, final_state, h0, chunk_states, scale, kernel)
    L.check(L.lib().harts_kda_fwd(plan.handle, ctypes.byref(a), _stream(stream)), "harts_kda_fwd")
    return o, states, final_state, chunk_states


def kda_bwd(plan: Plan, q, k, v, g, beta, d_o, *, states, chunk_states, d_final=None,
            h0=None, dh0=None, scale=1.0, grads=None, workspace=None,
            kernel=L.HARTS_KERNEL_AUTO, stream=None, phase="all"):
    """harts_kda_bwd (phase "all"), harts_kda_bwd_state ("state"), harts_kda_bwd_grad
    ("grad"), or harts_kda_bwd_static ("static": no workspace, the library's own scratch).
    Returns dict(dq, dk, dv, dg, dbeta[, dh0])."""
    import torch
    C, H, dk = q.shape
    dv = v.shape[2]
    dev = q.device
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dg=torch.empty_like(g), dbeta=torch.empty_like(beta))
    nb = plan.bwd_workspace_bytes(H, dk, dv)
    if workspace is None and phase != "static":
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    info = plan.info
    _need("d_o", d_o, (C, H, dv), q.dtype, device=dev)
    per = H * dk * dv * 4
    _need("d_final", d_final, None, torch.float32, info["n_seq"] * per, dev)
    _need("dh0", dh0, None, torch.float32, info["n_roots"] * per, dev)
    for n, ref in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta)):
        _need(n, grads[n], tuple(ref.shape), q.dtype, device=dev)
    if phase != "static":
        _need("workspace", workspace, nbytes=nb, device=dev)
    a = L.BwdArgs()
    a.fwd = _fwd_args(plan, q, k, v, g, beta, None, states, None, h0, chunk_states, scale, kernel)
    a.d_o = d_o.data_ptr()
    a.d_final = None if d_final is None else d_final.data_ptr()
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        setattr(a, n, grads[n].data_ptr())
    a.dh0 = None if dh0 is None else dh0.data_ptr()
    a.workspace = None if workspace is None else workspace.data_ptr()
    a.workspace_bytes = 0 if workspace is None else workspace.numel()
    fn = {"all": "harts_kda_bwd", "state": "harts_kda_bwd_state", "grad": "harts_kda_bwd_grad",
          "static": "harts_kda_bwd_static"}[phase]
    L.check(getattr(L.lib(), fn)(plan.handle, ctypes.byref(a), _stream(stream)), fn)
    if dh0 is not None:
        grads["dh0"] = dh0
    return grads


def _conv_args(x, weight, bias, y, activation):
    C, ch = x.shape[0], int(x.numel() // x.shape[0])
    a = L.ConvFwdArgs()
    a.channels, a.width = ch, int(weight.shape[1])
    a.dtype = dtype_code(x.dtype)
    a.activation = {"none": 0, "silu": 1}[activation]
    for n, t in dict(x=x, weight=weight, bias=bias, y=y).items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        setattr(a, n, None if t is None else t.data_ptr())
    return a


def conv_fwd(plan: Plan, x, weight, bias=None, *, activation="none", y=None, stream=None):
    """harts_conv_fwd.  x: [C, ...] compact rows (channels = the rest, flattened);
    weight: [channels, w] fp32; bias: [channels] fp32 or None.  Returns y like x."""
    import torch
    if y is None:
        y = torch.empty_like(x)
    a = _conv_args(x, weight, bias, y, activation)
    L.check(L.lib().harts_conv_fwd(plan.handle, ctypes.byref(a), _stream(stream)), "harts_conv_fwd")
    return y


def conv_bwd(plan: Plan, x, weight, bias, dy, *, activation="none", dx=None, dweight=None, dbias=None,
             workspace=None, stream=None):
    """harts_conv_bwd.  Returns (dx, dweight, dbias); dbias is None when bias is None."""
    import torch
    if dx is None:
        dx = torch.empty_like(x)
    if dweight is None:
        dweight = torch.empty_like(weight)
    if dbias is None and bias is not None:
        dbias = torch.empty_like(bias)
    b = L.ConvBwdArgs()
    b.fwd = _conv_args(x, weight, bias, None, activation)
    nb = int(L.lib().harts_conv_bwd_workspace_bytes(plan.handle, b.fwd.channels, b.fwd.width))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=x.device)
    b.dy, b.dx, b.dweight = dy.data_ptr(), dx.data_ptr(), dweight.data_ptr()
    b.dbias = None if dbias is None else dbias.data_ptr()
    b.workspace, b.workspace_bytes = workspace.data_ptr(), workspace.numel()
    L.check(L.lib().harts_conv_bwd(plan.handle, ctypes.byref(b), _stream(stream)), "harts_conv_bwd")
    return dx, dweight, dbias


def semantic_map(plan: Plan):
    """harts_plan_semantic_map: numpy (sem_row [S], row_ptr [C+1], row_sem [S]) int32."""
    C, S = plan.info["C"], plan.info["S"]
    sem_row = np.zeros(max(S, 1), np.int32)
    row_ptr = np.zeros(C + 1, np.int32)
    row_sem = np.zeros(max(S, 1), np.int32)
    L.check(L.lib().harts_plan_semantic_map(plan.handle, sem_row.ctypes.data_as(L._pi32),
                                            row_ptr.ctypes.data_as(L._pi32), row_sem.ctypes.data_as(L._pi32)),
            "harts_plan_semantic_map")
    return sem_row[:S], row_ptr, row_sem[:S]


def _lp_args(logits, row_ptr, row_sem, target, lse, logp):
    a = L.LogprobFwdArgs()
    a.C, a.V = logits.shape
    a.dtype = dtype_code(logits.dtype)
    a.S = target.numel()
    for n, t in dict(logits=logits, row_ptr=row_ptr, row_sem=row_sem, target=target, lse=lse, logp=logp).items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
        setattr(a, n, None if t is None else t.data_ptr())
    return a


def logprob_fwd(logits, row_ptr, row_sem, target, *, lse=None, logp=None, stream=None):
    """harts_logprob_fwd: returns (logp [S] fp32, lse [C] fp32)."""
    import torch
    if lse is None:
        lse = torch.empty(logits.shape[0], dtype=torch.float32, device=logits.device)
    if logp is None:
        logp = torch.empty(target.numel(), dtype=torch.float32, device=logits.device)
    a = _lp_args(logits, row_ptr, row_sem, target, lse, logp)
    L.check(L.lib().harts_logprob_fwd(ctypes.byref(a), _stream(stream)), "harts_logprob_fwd")
    return logp, lse


def logprob_bwd(logits, row_ptr, row_sem, target, lse, dlogp, *, dlogits=None, stream=None):
    """harts_logprob_bwd: returns dlogits like logits."""
    import torch
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    b = L.LogprobBwdArgs()
    b.fwd = _lp_args(logits, row_ptr, row_sem, target, lse, None)
    b.dlogp, b.dlogits = dlogp.data_ptr(), dlogits.data_ptr()
    L.check(L.lib().harts_logprob_bwd(ctypes.byref(b), _stream(stream)), "harts_logprob_bwd")
    return dlogits


def attn_fwd(plan: Plan, q, k, v, *, scale=None, o=None, lse=None, stream=None):
    """harts_attn_fwd: branch attention over the compact layout.  q, k, v: [C, H, d]
    bf16 (d = 128).  Returns (o [C, H, d] bf16, lse [C, H] fp32)."""
    import torch
    C, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((C, H), dtype=torch.float32, device=q.device)
    for n, t in dict(q=q, k=k, v=v, o=o, lse=lse).items():
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    a = _attn_args(q, k, v, o, lse, scale)
    L.check(L.lib().harts_attn_fwd(plan.handle, ctypes.byref(a), _stream(stream)), "harts_attn_fwd")
    return o, lse


def _attn_args(q, k, v, o, lse, scale):
    C, H, d = q.shape
    a = L.AttnFwdArgs()
    a.H, a.d, a.dtype = H, d, dtype_code(q.dtype)
    a.scale = float(d ** -0.5 if scale is None else scale)
    a.q, a.k, a.v, a.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    a.lse = None if lse is None else lse.data_ptr()
    return a


def attn_bwd(plan: Plan, q, k, v, o, lse, d_o, *, scale=None, dq=None, dk=None, dv=None, workspace=None,
             stream=None):
    """harts_attn_bwd: returns (dq, dk, dv) like q, from the forward's o and lse."""
    import torch
    for n, t in dict(q=q, k=k, v=v, o=o, lse=lse, d_o=d_o).items():
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    b = L.AttnBwdArgs()
    b.fwd = _attn_args(q, k, v, o, lse, scale)
    nb = int(L.lib().harts_attn_bwd_workspace_bytes(plan.handle, q.shape[1]))
    if workspace is None:
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    b.d_o, b.dq, b.dk, b.dv = d_o.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    b.workspace, b.workspace_bytes = workspace.data_ptr(), workspace.numel()
    L.check(L.lib().harts_attn_bwd(plan.handle, ctypes.byref(b), _stream(stream)), "harts_attn_bwd")
    return dq, dk, dv
