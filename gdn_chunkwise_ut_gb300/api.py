"""Python front end of libkkt: torch tensors in, the C ABI underneath.

``kkt_solve_fwd`` checks shapes and dtypes, allocates outputs with torch when
none are given, and passes raw device pointers and the current CUDA stream to
``kkt_solve_fwd_ex`` in libkkt.so.  Every step of the computation runs in the
library's CUDA kernels.
"""
from __future__ import annotations

import os

import torch

from . import _lib

_IO = {torch.bfloat16: _lib.KKT_IO_BF16, torch.float32: _lib.KKT_IO_F32}
_T_FLAG = {torch.float32: 0, torch.float16: _lib.KKT_T_OUT_F16}


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype, shape, host: bool = False):
    if not isinstance(t, torch.Tensor) or t.is_cuda != (not host):
        raise ValueError(f"{name} must be a {'host (CPU)' if host else 'CUDA'} tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_WORKSPACES = {}


def _workspace(device: torch.device) -> torch.Tensor:
    """The per-device scratch buffer the default calls share (stream-ordered use)."""
    key = (device.type, device.index)
    ws = _WORKSPACES.get(key)
    if ws is None:
        ws = torch.zeros(_lib.KKT_WORKSPACE_BYTES // 4, dtype=torch.int32, device=device)
        _WORKSPACES[key] = ws
    return ws


def kkt_solve_fwd(k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, C: int,
                  cu_seqlens: torch.Tensor | None = None, *, T_out=None, W_out=None, U_out=None,
                  kernel: str = "auto", workspace="auto", stream=None, materialize_T: bool = True,
                  T_dtype=torch.float32, g: torch.Tensor | None = None, check: bool | None = None):
    """UT transform of every chunk: returns (T_out, W, U).

    ``materialize_T=False`` computes T but does not write it: the call returns (None, W, U) and
    moves 4C bytes less per token and head.  ``T_dtype=torch.float16`` writes T rounded to fp16
    (2C bytes per token and head); W and U are the same as with fp32 T.  ``g`` [B, T, H] fp32 (the
    per-token log decays) selects the gated variant: A = I + strictLower(diag(beta)(Gamma o K K^T))
    with Gamma[i][j] = exp(g_{j+1} + ... + g_i) inside each chunk.

    k [B, T, H, dk] and v [B, T, H, dv] (bf16, or fp32 for the fp32-I/O path),
    beta [B, T, H] fp32.  With ``cu_seqlens`` (int32 [N+1] on the device) the
    tensors are [1, T, H, .] and hold N packed sequences.  T_out is [B, T, H, C]
    of ``T_dtype``; W and U have k's dtype.  ``kernel`` is "auto", "simt" or "tc".
    ``workspace``: "auto" uses a cached per-device scratch buffer (dynamic tile
    scheduling; calls on concurrent streams should pass their own), a CUDA tensor
    of at least KKT_WORKSPACE_BYTES, zero-filled before its first use (every call
    leaves it zero), or None for the fixed round-robin schedule.
    ``check=True`` (default: the environment variable KKT_CHECK=1) is the checked mode: the call
    synchronises the stream, reads and clears the device status word, and raises KktError when the
    kernel recorded an error (a malformed cu_seqlens, an expired bounded wait).
    """
    if k.dim() != 4 or v.dim() != 4 or beta.dim() != 3:
        raise ValueError("expected k [B,T,H,dk], v [B,T,H,dv], beta [B,T,H]")
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    io = _IO.get(k.dtype)
    if io is None:
        raise ValueError(f"unsupported dtype {k.dtype}")
    t_flag = _T_FLAG.get(T_dtype)
    if t_flag is None:
        raise ValueError(f"T_dtype must be torch.float32 or torch.float16, got {T_dtype}")
    _check(k, "k", k.dtype, (Bt, T, H, dk))
    _check(v, "v", k.dtype, (Bt, T, H, dv))
    _check(beta, "beta", torch.float32, (Bt, T, H))
    if g is not None:
        _check(g, "g", torch.float32, (Bt, T, H))
    if cu_seqlens is not None:
        if Bt != 1:
            raise ValueError("with cu_seqlens the batch dimension must be 1")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        B = cu_seqlens.shape[0] - 1
        cu_ptr = cu_seqlens.data_ptr()
    else:
        B, cu_ptr = Bt, None
    dev = k.device
    if not materialize_T:
        if T_out is not None:
            raise ValueError("T_out given with materialize_T=False")
    elif T_out is None:
        T_out = torch.empty((Bt, T, H, C), device=dev, dtype=T_dtype)
    if W_out is None:
        W_out = torch.empty((Bt, T, H, dk), device=dev, dtype=k.dtype)
    if U_out is None:
        U_out = torch.empty((Bt, T, H, dv), device=dev, dtype=k.dtype)
    if materialize_T:
        _check(T_out, "T_out", T_dtype, (Bt, T, H, C))
    _check(W_out, "W_out", k.dtype, (Bt, T, H, dk))
    _check(U_out, "U_out", k.dtype, (Bt, T, H, dv))
    kern = _lib.KERNELS.get(kernel)
    if kern is None:
        raise ValueError(f"kernel must be one of {sorted(_lib.KERNELS)}")
    if isinstance(workspace, str) and workspace == "auto":
        workspace = _workspace(dev)
    if workspace is None:
        ws_ptr, ws_bytes = None, 0
    else:
        if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor, 'auto' or None")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    t_ptr = T_out.data_ptr() if materialize_T else None
    if g is None:
        rc = _lib.lib().kkt_solve_fwd_ex(k.data_ptr(), v.data_ptr(), beta.data_ptr(), cu_ptr, B, T, H, dk, dv, C,
                                         t_ptr, W_out.data_ptr(), U_out.data_ptr(), io | t_flag, kern, ws_ptr,
                                         ws_bytes, _stream_handle(stream))
    else:
        rc = _lib.lib().kkt_solve_fwd_gated(k.data_ptr(), v.data_ptr(), beta.data_ptr(), g.data_ptr(), cu_ptr, B, T,
                                            H, dk, dv, C, t_ptr, W_out.data_ptr(), U_out.data_ptr(), io | t_flag,
                                            kern, ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != _lib.KKT_OK:
        raise _lib.KktError(rc, "kkt_solve_fwd")
    if check is None:
        check = os.environ.get("KKT_CHECK", "0") == "1"
    if check:
        st = device_status(stream)
        if st != _lib.KKT_OK:
            raise _lib.KktError(st, "kkt_solve_fwd (device)")
    return T_out, W_out, U_out


def gdn_chunk_state_fwd(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, u: torch.Tensor, C: int = 64, *,
                        g: torch.Tensor | None = None, initial_state: torch.Tensor | None = None, scale=None,
                        cu_seqlens: torch.Tensor | None = None, output_final_state: bool = True, o=None,
                        final_state=None, stream=None, check: bool | None = None):
    """The chunk state recurrence and output that consume kkt_solve's W and U~: returns (o, final_state).

    q, k, w [B, T, H, dk] and u [B, T, H, dv] bf16 (w, u: the W and U of ``kkt_solve_fwd`` on the same k,
    beta, g, cu_seqlens and C); ``g`` [B, T, H] fp32 log decays or None; ``initial_state`` [N, H, dk, dv]
    fp32 or None (zero), N the number of sequences; ``scale`` defaults to dk ** -0.5.  o is [B, T, H, dv]
    bf16; final_state [N, H, dk, dv] fp32, or None when ``output_final_state`` is False.  The recurrence
    is S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T, o_t = scale S_t^T q_t, with
    alpha_t = exp(g_t); the library computes it chunk by chunk (see include/kkt.h).
    """
    if q.dim() != 4 or k.dim() != 4 or w.dim() != 4 or u.dim() != 4:
        raise ValueError("expected q, k, w [B,T,H,dk] and u [B,T,H,dv]")
    Bt, T, H, dk = k.shape
    dv = u.shape[-1]
    for name, x, d in (("q", q, dk), ("k", k, dk), ("w", w, dk), ("u", u, dv)):
        _check(x, name, torch.bfloat16, (Bt, T, H, d))
    if g is not None:
        _check(g, "g", torch.float32, (Bt, T, H))
    if cu_seqlens is not None:
        if Bt != 1:
            raise ValueError("with cu_seqlens the batch dimension must be 1")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        N, cu_ptr = cu_seqlens.shape[0] - 1, cu_seqlens.data_ptr()
    else:
        N, cu_ptr = Bt, None
    dev = k.device
    if initial_state is not None:
        _check(initial_state, "initial_state", torch.float32, (N, H, dk, dv))
    if o is None:
        o = torch.empty((Bt, T, H, dv), device=dev, dtype=torch.bfloat16)
    _check(o, "o", torch.bfloat16, (Bt, T, H, dv))
    if output_final_state:
        if final_state is None:
            final_state = torch.empty((N, H, dk, dv), device=dev, dtype=torch.float32)
        _check(final_state, "final_state", torch.float32, (N, H, dk, dv))
    else:
        final_state = None
    if scale is None:
        scale = dk ** -0.5
    rc = _lib.lib().gdn_chunk_state_fwd(q.data_ptr(), k.data_ptr(), w.data_ptr(), u.data_ptr(),
                                        None if g is None else g.data_ptr(),
                                        None if initial_state is None else initial_state.data_ptr(), cu_ptr,
                                        N, T, H, dk, dv, C, float(scale), o.data_ptr(),
                                        None if final_state is None else final_state.data_ptr(),
                                        _stream_handle(stream))
    if rc != _lib.KKT_OK:
        raise _lib.KktError(rc, "gdn_chunk_state_fwd")
    if check is None:
        check = os.environ.get("KKT_CHECK", "0") == "1"
    if check:
        st = device_status(stream)
        if st != _lib.KKT_OK:
            raise _lib.KktError(st, "gdn_chunk_state_fwd (device)")
    return o, final_state


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state: bool = False,
                           cu_seqlens=None, *, C: int = 64, stream=None):
    """The forward pass of Gated DeltaNet chunked prefill, in the argument order of the FlashQLA API:
    kkt_solve (W and U~ only, T not written) then the chunk state recurrence and output.  ``g`` may
    be None (the ungated delta rule).  Returns (o, final_state or None)."""
    _, W, U = kkt_solve_fwd(k, v, beta, C, cu_seqlens, materialize_T=False, g=g, stream=stream)
    return gdn_chunk_state_fwd(q, k, W, U, C, g=g, initial_state=initial_state, scale=scale, cu_seqlens=cu_seqlens,
                               output_final_state=output_final_state, stream=stream)


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status word."""
    return int(_lib.lib().kkt_device_status(_stream_handle(stream)))


def select_kernel(dk: int, dv: int, C: int, io: str = "bf16", kernel: str = "auto") -> str:
    """Which kernel a call would run ("simt" / "tc"); raises KktError if unsupported."""
    iod = _lib.KKT_IO_F32 if io == "f32" else _lib.KKT_IO_BF16
    r = _lib.lib().kkt_select_kernel(dk, dv, C, iod, _lib.KERNELS[kernel])
    if r < 0:
        raise _lib.KktError(-r, "kkt_select_kernel")
    return {_lib.KKT_KERNEL_SIMT: "simt", _lib.KKT_KERNEL_TC: "tc"}[r]


def host_workspace_bytes(B: int, T: int, H: int, dk: int, dv: int, C: int, *, dtype=torch.bfloat16,
                         T_dtype=torch.float32, gated: bool = False, varlen: bool = False, pieces: int = 8) -> int:
    """Device workspace bytes of ``kkt_solve_fwd_host`` for these sizes (no CUDA call)."""
    io = _IO.get(dtype)
    if io is None:
        raise ValueError(f"unsupported dtype {dtype}")
    n = _lib.lib().kkt_host_workspace_bytes(B, T, H, dk, dv, C, io | _T_FLAG[T_dtype], int(gated), int(varlen),
                                            int(pieces))
    if n == 0:
        raise ValueError("invalid sizes or pieces")
    return int(n)


def kkt_solve_fwd_host(k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, C: int, cu_seqlens=None, *,
                       T_out=None, W_out=None, U_out=None, g: torch.Tensor | None = None,
                       materialize_T: bool = True, T_dtype=torch.float32, kernel: str = "auto", pieces: int = 8,
                       workspace: torch.Tensor | None = None, device="cuda", stream=None, sync: bool = True):
    """kkt_solve on HOST tensors through the C ABI (kkt_solve_fwd_host): the library copies k, v, beta
    (and g) to the device, runs kkt_solve and copies T, W and U back, pipelined in ``pieces`` parts
    of the token axis.  The results equal those of ``kkt_solve_fwd`` on the device.

    k, v, beta, g and the outputs are CPU tensors (pinned memory lets the copies overlap; the
    outputs are allocated pinned when not given).  ``cu_seqlens``: None, or the B + 1 sequence
    offsets as a CPU int32 tensor or a list.  ``workspace``: a CUDA uint8 tensor of at least
    ``host_workspace_bytes(...)`` bytes (allocated when None; pass one to reuse it).  ``sync``
    waits for the copies back before returning.  Returns (T_out, W, U) on the host.
    """
    if k.dim() != 4 or v.dim() != 4 or beta.dim() != 3:
        raise ValueError("expected k [B,T,H,dk], v [B,T,H,dv], beta [B,T,H]")
    Bt, T, H, dk = k.shape
    dv = v.shape[-1]
    io = _IO.get(k.dtype)
    if io is None:
        raise ValueError(f"unsupported dtype {k.dtype}")
    t_flag = _T_FLAG.get(T_dtype)
    if t_flag is None:
        raise ValueError(f"T_dtype must be torch.float32 or torch.float16, got {T_dtype}")
    _check(k, "k", k.dtype, (Bt, T, H, dk), host=True)
    _check(v, "v", k.dtype, (Bt, T, H, dv), host=True)
    _check(beta, "beta", torch.float32, (Bt, T, H), host=True)
    if g is not None:
        _check(g, "g", torch.float32, (Bt, T, H), host=True)
    cu_host = None
    if cu_seqlens is not None:
        if Bt != 1:
            raise ValueError("with cu_seqlens the batch dimension must be 1")
        cu_host = torch.as_tensor(cu_seqlens, dtype=torch.int32).contiguous()
        if cu_host.is_cuda or cu_host.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D host int32 tensor or a list")
        B = cu_host.shape[0] - 1
    else:
        B = Bt
    pin = torch.cuda.is_available()
    if not materialize_T:
        if T_out is not None:
            raise ValueError("T_out given with materialize_T=False")
    elif T_out is None:
        T_out = torch.empty((Bt, T, H, C), dtype=T_dtype, pin_memory=pin)
    if W_out is None:
        W_out = torch.empty((Bt, T, H, dk), dtype=k.dtype, pin_memory=pin)
    if U_out is None:
        U_out = torch.empty((Bt, T, H, dv), dtype=k.dtype, pin_memory=pin)
    if materialize_T:
        _check(T_out, "T_out", T_dtype, (Bt, T, H, C), host=True)
    _check(W_out, "W_out", k.dtype, (Bt, T, H, dk), host=True)
    _check(U_out, "U_out", k.dtype, (Bt, T, H, dv), host=True)
    kern = _lib.KERNELS.get(kernel)
    if kern is None:
        raise ValueError(f"kernel must be one of {sorted(_lib.KERNELS)}")
    need = host_workspace_bytes(B, T, H, dk, dv, C, dtype=k.dtype, T_dtype=T_dtype, gated=g is not None,
                                varlen=cu_host is not None, pieces=pieces)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
        if stream is not None:  # the buffer is freed on return, in use on `stream` until the call ends
            workspace.record_stream(stream)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    rc = _lib.lib().kkt_solve_fwd_host(k.data_ptr(), v.data_ptr(), beta.data_ptr(),
                                       None if g is None else g.data_ptr(),
                                       None if cu_host is None else cu_host.data_ptr(), B, T, H, dk, dv, C,
                                       T_out.data_ptr() if materialize_T else None, W_out.data_ptr(),
                                       U_out.data_ptr(), io | t_flag, kern, int(pieces), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != _lib.KKT_OK:
        raise _lib.KktError(rc, "kkt_solve_fwd_host")
    if sync:
        (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return T_out, W_out, U_out


class HostRunner:
    """End-to-end calls on host tensors through ``kkt_solve_fwd_host`` (the C ABI's host-buffer entry
    point), with the device workspace and the pinned host outputs allocated once.

    Each call copies the inputs in, runs kkt_solve and copies T, W and U back, pipelined by the
    library in ``pieces`` parts of the token axis (whole sequences, or chunk-aligned parts of one)
    on its own copy streams and the current stream.  The results are those of one call on the whole
    batch.  ``sync=True`` waits for the copies.
    """

    def __init__(self, B, T, H, dk, dv, C, *, dtype=torch.bfloat16, cu_seqlens=None,
                 kernel="auto", device="cuda", materialize_T: bool = True, T_dtype=torch.float32,
                 gated: bool = False, pieces: int = 8):
        self.C, self.kernel, self.materialize_T, self.T_dtype = C, kernel, materialize_T, T_dtype
        self.pieces, self.gated = int(pieces), gated
        self.cu = None if cu_seqlens is None else torch.as_tensor(
            [int(x) for x in cu_seqlens], dtype=torch.int32)
        nseq = B if self.cu is None else self.cu.shape[0] - 1
        self.shape = (B, T, H)
        self.sizes = (dk, dv)
        self.dtype = dtype
        self.workspace = torch.empty(
            host_workspace_bytes(nseq, T, H, dk, dv, C, dtype=dtype, T_dtype=T_dtype, gated=gated,
                                 varlen=self.cu is not None, pieces=self.pieces),
            dtype=torch.uint8, device=device)
        self.T_host = torch.empty((B, T, H, C), dtype=T_dtype, pin_memory=True) if materialize_T else None
        self.W_host = torch.empty((B, T, H, dk), dtype=dtype, pin_memory=True)
        self.U_host = torch.empty((B, T, H, dv), dtype=dtype, pin_memory=True)

    @property
    def h2d_bytes(self) -> int:
        B, T, H = self.shape
        dk, dv = self.sizes
        es = torch.empty((), dtype=self.dtype).element_size()
        return B * T * H * ((dk + dv) * es + 4 + (4 if self.gated else 0))

    @property
    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.T_host, self.W_host, self.U_host) if t is not None)

    def __call__(self, k_host, v_host, beta_host, sync: bool = True, g_host=None):
        if (g_host is not None) != self.gated:
            raise ValueError("g_host must be given exactly when the runner is gated")
        return kkt_solve_fwd_host(k_host, v_host, beta_host, self.C, self.cu, T_out=self.T_host, W_out=self.W_host,
                                  U_out=self.U_host, g=g_host, materialize_T=self.materialize_T,
                                  T_dtype=self.T_dtype, kernel=self.kernel, pieces=self.pieces,
                                  workspace=self.workspace, sync=sync)
