"""Python binding of the C ABI: argument marshalling only.

Each function takes CUDA tensors, passes their device pointers, leading
dimensions and the current torch stream to libtee.so, and returns the output
tensors. No step of the computation runs in Python or PyTorch: the library
kernels do all of it, and a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
from typing import Dict, List, Optional, Sequence

import torch

from . import _lib
from ._lib import (CacheLayout, FillDesc, FillLayer, GateDesc, StepBuffers, check, load)

_DT = {torch.float32: _lib.TEE_F32, torch.float16: _lib.TEE_F16, torch.bfloat16: _lib.TEE_BF16}
_RULE = {"per_token": _lib.TEE_RULE_PER_TOKEN, "batch_all": _lib.TEE_RULE_BATCH_ALL}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _mat(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with contiguous rows")
    return t


def _vec(t: Optional[torch.Tensor], name: str) -> Optional[torch.Tensor]:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


class Workspace:
    """Device scratch for the calls. Grows on demand; a new buffer is
    zero-filled once through tee_workspace_init, as the ABI requires."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int):
        nbytes = max(int(nbytes), _lib.WS_HEADER_BYTES)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
            check("tee_workspace_init", load().tee_workspace_init(_ptr(self.buf), nbytes, _stream(self.device)))
        return _ptr(self.buf), self.buf.numel()

    def device_error(self):
        """(code, detail) of the first device fault recorded; synchronises the stream."""
        if self.buf is None:
            return 0, 0
        code, detail = ctypes.c_int32(0), ctypes.c_int32(0)
        st = load().tee_get_device_error(_ptr(self.buf), ctypes.byref(code), ctypes.byref(detail),
                                         _stream(self.device))
        if st not in (_lib.TEE_OK, _lib.TEE_ERR_DEVICE):
            check("tee_get_device_error", st)
        return code.value, detail.value

    def check_wait_timeout(self, limit_us: int = 1000):
        """Run the library's bounded wait against a barrier that nothing completes
        (tee_check_wait_timeout): the wait records a time-out here and returns."""
        wp, wn = self.get(_lib.WS_HEADER_BYTES)
        check("tee_check_wait_timeout", load().tee_check_wait_timeout(wp, int(limit_us), _stream(self.device)))

    def clear_error(self):
        if self.buf is not None:
            check("tee_clear_device_error", load().tee_clear_device_error(_ptr(self.buf), _stream(self.device)))


def exit_gate(h_cur: torch.Tensor, threshold: float, *, h_prev: Optional[torch.Tensor] = None,
              w_down: Optional[torch.Tensor] = None, w_up: Optional[torch.Tensor] = None,
              gamma: Optional[torch.Tensor] = None, b_down: Optional[torch.Tensor] = None,
              b_up: Optional[torch.Tensor] = None, rule: str = "per_token", eps: float = 1e-5,
              ws: Optional[Workspace] = None, out: Optional[Dict[str, torch.Tensor]] = None):
    """Cosine gate when ``h_prev`` is given, else TIDE router gate (``w_down``,
    ``w_up``). Returns (score f32[n], mask u8[n], batch_flag i32[1])."""
    lib = load()
    h_cur = _mat(h_cur, "h_cur")
    n, d = h_cur.shape
    cosine = h_prev is not None
    desc = GateDesc(mode=_lib.TEE_GATE_COSINE if cosine else _lib.TEE_GATE_ROUTER, rule=_RULE[rule],
                    dtype=_DT[h_cur.dtype], d=d, bottleneck=0 if cosine else int(w_down.shape[0]),
                    threshold=float(threshold), eps=float(eps))
    if cosine:
        _mat(h_prev, "h_prev")
    else:
        _mat(w_down, "w_down")
        _vec(w_up, "w_up")
    out = out or {}
    score = out["score"] if "score" in out else torch.empty(n, dtype=torch.float32, device=h_cur.device)
    mask = out["mask"] if "mask" in out else torch.empty(n, dtype=torch.uint8, device=h_cur.device)
    flag = out["flag"] if "flag" in out else torch.empty(1, dtype=torch.int32, device=h_cur.device)
    ws = ws or Workspace(h_cur.device)
    wp, wn = ws.get(lib.tee_exit_gate_workspace_size(ctypes.byref(desc), n))
    st = lib.tee_exit_gate(ctypes.byref(desc), n, _ptr(h_cur), h_cur.stride(0),
                           _ptr(h_prev), h_prev.stride(0) if cosine else 0,
                           _ptr(_vec(gamma, "gamma")), _ptr(w_down), _ptr(_vec(b_down, "b_down")),
                           _ptr(w_up), _ptr(_vec(b_up, "b_up")), _ptr(score), _ptr(mask), _ptr(flag),
                           wp, wn, _stream(h_cur.device))
    check("tee_exit_gate", st)
    return score, mask, flag


def exit_compact(mask: torch.Tensor, *, pos_in: Optional[torch.Tensor] = None, h: Optional[torch.Tensor] = None,
                 ws: Optional[Workspace] = None, out: Optional[Dict[str, torch.Tensor]] = None,
                 with_pos: bool = True) -> Dict[str, torch.Tensor]:
    """Stable split by ``mask``; gathers the continuing rows of ``h`` when given."""
    lib = load()
    mask = _vec(mask, "mask")
    n = mask.numel()
    dev = mask.device
    out = dict(out or {})
    for k in ("cont_rows", "exit_rows") + (("cont_pos", "exit_pos") if with_pos else ()):
        if k not in out:
            out[k] = torch.empty(n, dtype=torch.int32, device=dev)
    if "counts" not in out:
        out["counts"] = torch.empty(2, dtype=torch.int32, device=dev)
    d, dt, ldi, ldc = 0, _lib.TEE_BF16, 0, 0
    if h is not None:
        _mat(h, "h")
        d = h.shape[1]
        dt = _DT[h.dtype]
        if "h_cont" not in out:
            out["h_cont"] = torch.empty((n, d), dtype=h.dtype, device=dev)
        ldi, ldc = h.stride(0), out["h_cont"].stride(0)
    ws = ws or Workspace(dev)
    wp, wn = ws.get(lib.tee_exit_compact_workspace_size(n))
    st = lib.tee_exit_compact(n, _ptr(mask), _ptr(_vec(pos_in, "pos_in")), _ptr(h), ldi, d, dt,
                              _ptr(out["cont_rows"]), _ptr(out["exit_rows"]), _ptr(out.get("cont_pos")),
                              _ptr(out.get("exit_pos")), _ptr(out.get("h_cont")), ldc, _ptr(out["counts"]),
                              wp, wn, _stream(dev))
    check("tee_exit_compact", st)
    return out


def exit_compact_scatter(mask: torch.Tensor, h: torch.Tensor, out: torch.Tensor, *,
                         pos_in: Optional[torch.Tensor] = None, gather: bool = True,
                         ws: Optional[Workspace] = None, res: Optional[Dict[str, torch.Tensor]] = None,
                         with_pos: bool = True) -> Dict[str, torch.Tensor]:
    """exit_compact (gathering the continuing rows of ``h`` when ``gather``) and the
    exit scatter out[pos_in[r] or r] = h[r] of every exiting row r, in one launch."""
    lib = load()
    mask = _vec(mask, "mask")
    n = mask.numel()
    dev = mask.device
    _mat(h, "h")
    _mat(out, "out")
    d = h.shape[1]
    res = dict(res or {})
    for k in ("cont_rows", "exit_rows") + (("cont_pos", "exit_pos") if with_pos else ()):
        if k not in res:
            res[k] = torch.empty(n, dtype=torch.int32, device=dev)
    if "counts" not in res:
        res["counts"] = torch.empty(2, dtype=torch.int32, device=dev)
    if gather and "h_cont" not in res:
        res["h_cont"] = torch.empty((n, d), dtype=h.dtype, device=dev)
    h_cont = res.get("h_cont") if gather else None
    ws = ws or Workspace(dev)
    wp, wn = ws.get(lib.tee_exit_compact_workspace_size(n))
    st = lib.tee_exit_compact_scatter(n, _ptr(mask), _ptr(_vec(pos_in, "pos_in")), _ptr(h), h.stride(0), d,
                                      _DT[h.dtype], _ptr(res["cont_rows"]), _ptr(res["exit_rows"]),
                                      _ptr(res.get("cont_pos")), _ptr(res.get("exit_pos")), _ptr(h_cont),
                                      h_cont.stride(0) if h_cont is not None else 0, _ptr(out), out.stride(0),
                                      out.shape[0], _ptr(res["counts"]), wp, wn, _stream(dev))
    check("tee_exit_compact_scatter", st)
    return res


def exit_gate_compact_scatter(h_cur: torch.Tensor, h_prev: torch.Tensor, threshold: float, out: torch.Tensor, *,
                              rule: str = "per_token", pos_in: Optional[torch.Tensor] = None, gather: bool = True,
                              ws: Optional[Workspace] = None, res: Optional[Dict[str, torch.Tensor]] = None,
                              with_pos: bool = True) -> Dict[str, torch.Tensor]:
    """Cosine exit gate, compaction (continuing rows of ``h_cur`` gathered when
    ``gather``) and the exit scatter out[pos_in[r] or r] = h_cur[r], one launch for
    up to 128 tokens. Returns score, mask, flag, counts and the row lists."""
    lib = load()
    h_cur = _mat(h_cur, "h_cur")
    _mat(h_prev, "h_prev")
    _mat(out, "out")
    n, d = h_cur.shape
    dev = h_cur.device
    desc = GateDesc(mode=_lib.TEE_GATE_COSINE, rule=_RULE[rule], dtype=_DT[h_cur.dtype], d=d, bottleneck=0,
                    threshold=float(threshold), eps=1e-5)
    res = dict(res or {})
    if "score" not in res:
        res["score"] = torch.empty(n, dtype=torch.float32, device=dev)
    if "mask" not in res:
        res["mask"] = torch.empty(n, dtype=torch.uint8, device=dev)
    if "flag" not in res:
        res["flag"] = torch.empty(1, dtype=torch.int32, device=dev)
    for k in ("cont_rows", "exit_rows") + (("cont_pos", "exit_pos") if with_pos else ()):
        if k not in res:
            res[k] = torch.empty(n, dtype=torch.int32, device=dev)
    if "counts" not in res:
        res["counts"] = torch.empty(2, dtype=torch.int32, device=dev)
    if gather and "h_cont" not in res:
        res["h_cont"] = torch.empty((n, d), dtype=h_cur.dtype, device=dev)
    h_cont = res.get("h_cont") if gather else None
    ws = ws or Workspace(dev)
    wp, wn = ws.get(lib.tee_exit_gate_compact_scatter_workspace_size(ctypes.byref(desc), n))
    st = lib.tee_exit_gate_compact_scatter(
        ctypes.byref(desc), n, _ptr(h_cur), h_cur.stride(0), _ptr(h_prev), h_prev.stride(0), None, None, None, None,
        None, _ptr(_vec(pos_in, "pos_in")), _ptr(res["score"]), _ptr(res["mask"]), _ptr(res["flag"]),
        _ptr(res["cont_rows"]), _ptr(res["exit_rows"]), _ptr(res.get("cont_pos")), _ptr(res.get("exit_pos")),
        _ptr(h_cont), h_cont.stride(0) if h_cont is not None else 0, _ptr(out), out.stride(0), out.shape[0],
        _ptr(res["counts"]), wp, wn, _stream(dev))
    check("tee_exit_gate_compact_scatter", st)
    return res


def exit_scatter(counts: torch.Tensor, exit_rows: torch.Tensor, exit_pos: torch.Tensor, h_src: torch.Tensor,
                 out: torch.Tensor, *, final_gamma: Optional[torch.Tensor] = None, eps: float = 1e-5,
                 n_max: Optional[int] = None, ws: Optional[Workspace] = None) -> torch.Tensor:
    """out[exit_pos[i]] = h_src[exit_rows[i]] (optionally RMSNorm * final_gamma) for i < counts[1]."""
    lib = load()
    _mat(h_src, "h_src")
    _mat(out, "out")
    n_max = h_src.shape[0] if n_max is None else int(n_max)
    ws = ws or Workspace(out.device)
    wp, wn = ws.get(lib.tee_exit_scatter_workspace_size(n_max))
    st = lib.tee_exit_scatter(n_max, _ptr(_vec(counts, "counts")), _ptr(_vec(exit_rows, "exit_rows")),
                              _ptr(_vec(exit_pos, "exit_pos")), _ptr(h_src), h_src.stride(0), _ptr(out),
                              out.stride(0), out.shape[0], h_src.shape[1], _DT[h_src.dtype],
                              _ptr(_vec(final_gamma, "final_gamma")), float(eps), wp, wn, _stream(out.device))
    check("tee_exit_scatter", st)
    return out


def cache_layout(cache: torch.Tensor) -> CacheLayout:
    """Layout of a [layers][seqs][kv_heads][positions][head_dim] cache tensor."""
    if cache.dim() != 5 or cache.stride(4) != 1:
        raise ValueError("cache must be 5-D [layers][seqs][kv_heads][positions][head_dim] with contiguous head_dim")
    s = cache.stride()
    L, S, H, P, _ = cache.shape
    return CacheLayout(s_layer=s[0], s_seq=s[1], s_head=s[2], s_pos=s[3], n_layers=L, n_seq=S, n_heads=H, max_pos=P)


class KVFill:
    """Prepared KV fill for a fixed set of filled layers.

    ``layers`` holds one dict per filled layer with CUDA tensors ``gamma``,
    ``wk``, ``wv`` (dense [d][kvw] or packed int4 [d/2][kvw]), optionally
    ``w_map`` [d][d] and, for int4, ``k_scale``, ``k_zero``, ``v_scale``,
    ``v_zero`` [d/group][kvw] fp16, plus the int ``cache_layer``. Model-family
    variants: ``k_bias``, ``v_bias`` [kvw] and ``k_norm`` [head_dim] tensors, and
    ``writes`` = "k" or "v" to fill only one of the caches. ``generic`` runs
    every call on the generic CUDA-core kernels (for checking the fused paths).
    """

    def __init__(self, layers: Sequence[Dict], *, d: int, n_kv_heads: int, head_dim: int, rope_base: float,
                 eps: float, dtype: torch.dtype, max_pos: int, int4: bool = False, group: int = 64,
                 early_weights: bool = False, generic: bool = False):
        self.lib = load()
        self.desc = FillDesc(d=d, n_kv_heads=n_kv_heads, head_dim=head_dim, rope_base=float(rope_base),
                             eps=float(eps), dtype=_DT[dtype], wfmt=_lib.TEE_W_INT4 if int4 else _lib.TEE_W_DENSE,
                             group=group, flags=(_lib.TEE_FILL_EARLY_WEIGHTS if early_weights else 0)
                             | (_lib.TEE_FILL_GENERIC if generic else 0))
        self.keep: List[torch.Tensor] = []
        arr = (FillLayer * max(1, len(layers)))()
        dev = None
        for i, L in enumerate(layers):
            def p(k):
                t = L.get(k)
                if t is None:
                    return None
                _vec(t, k)
                self.keep.append(t)
                return t.data_ptr()
            arr[i].w_map, arr[i].gamma, arr[i].wk, arr[i].wv = p("w_map"), p("gamma"), p("wk"), p("wv")
            arr[i].k_scale, arr[i].k_zero = p("k_scale"), p("k_zero")
            arr[i].v_scale, arr[i].v_zero = p("v_scale"), p("v_zero")
            arr[i].cache_layer = int(L["cache_layer"])
            arr[i].k_bias, arr[i].v_bias, arr[i].k_norm = p("k_bias"), p("v_bias"), p("k_norm")
            arr[i].writes = {None: 0, "kv": 0, "k": _lib.TEE_FILL_WRITE_K, "v": _lib.TEE_FILL_WRITE_V}[L.get("writes")]
            dev = L["gamma"].device
        self.layers = arr
        self.n_layers = len(layers)
        self.max_pos = int(max_pos)
        self.device = dev or torch.device("cuda")
        nbytes = self.lib.tee_kv_fill_prep_size(ctypes.byref(self.desc), self.n_layers, self.max_pos)
        if nbytes == 0:
            raise ValueError("invalid KV fill descriptor")
        self.prep = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        st = self.lib.tee_kv_fill_prepare(ctypes.byref(self.desc), self.n_layers, self.layers, self.max_pos,
                                          _ptr(self.prep), nbytes, _stream(self.device))
        check("tee_kv_fill_prepare", st)

    def workspace_bytes(self, n_max: int) -> int:
        return self.lib.tee_kv_fill_workspace_size(ctypes.byref(self.desc), self.n_layers, int(n_max))

    def __call__(self, h_split: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                 rows: Optional[torch.Tensor] = None, pos: Optional[torch.Tensor] = None, pos0: int = 0,
                 seq: Optional[torch.Tensor] = None, n_dev: Optional[torch.Tensor] = None,
                 n_max: Optional[int] = None, ws: Optional[Workspace] = None) -> None:
        _mat(h_split, "h_split")
        if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape:
            raise ValueError("k_cache and v_cache must share one layout")
        layout = cache_layout(k_cache)
        if n_max is None:
            n_max = rows.numel() if rows is not None else h_split.shape[0]
        ws = ws or Workspace(h_split.device)
        wp, wn = ws.get(self.workspace_bytes(n_max))
        st = self.lib.tee_kv_fill(ctypes.byref(self.desc), self.n_layers, self.layers, _ptr(self.prep),
                                  self.prep.numel(), int(n_max), _ptr(_vec(n_dev, "n_dev")), _ptr(h_split),
                                  h_split.stride(0), h_split.shape[0], _ptr(_vec(rows, "rows")),
                                  _ptr(_vec(pos, "pos")), int(pos0), _ptr(_vec(seq, "seq")), _ptr(k_cache),
                                  _ptr(v_cache), ctypes.byref(layout), wp, wn, _stream(h_split.device))
        check("tee_kv_fill", st)


class DecodeStep:
    """A whole decode step from host buffers to host buffers in one library call
    (tee_decode_step_run_host): the inputs' copies to the device, the cosine
    gate with compaction and exit scatter in one launch, the KV fill of the
    exiting tokens with ``fill`` (a prepared KVFill), and the results' copies
    back, all on the current stream. The device buffers are allocated here and
    kept; ``k_cache`` / ``v_cache`` are filled in place. Host tensors passed to
    ``run_host`` should be pinned for the copies to overlap."""

    def __init__(self, fill: "KVFill", *, n_max: int, d: int, threshold: float, dtype: torch.dtype,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, rule: str = "per_token", device=None):
        self.lib = load()
        dev = torch.device(device or k_cache.device)
        self.fill, self.n_max, self.d, self.dtype = fill, int(n_max), int(d), dtype
        self.gate = GateDesc(mode=_lib.TEE_GATE_COSINE, rule=_RULE[rule], dtype=_DT[dtype], d=self.d, bottleneck=0,
                             threshold=float(threshold), eps=1e-5)
        n = self.n_max
        i32 = dict(dtype=torch.int32, device=dev)
        self.t = {"h_prev": torch.empty(n, d, dtype=dtype, device=dev), "h_cur": torch.empty(n, d, dtype=dtype, device=dev),
                  "pos": torch.empty(n, **i32), "seq": torch.zeros(n, **i32),
                  "score": torch.empty(n, dtype=torch.float32, device=dev),
                  "mask": torch.empty(n, dtype=torch.uint8, device=dev), "flag": torch.empty(1, **i32),
                  "cont_rows": torch.empty(n, **i32), "exit_rows": torch.empty(n, **i32),
                  "cont_pos": torch.empty(n, **i32), "exit_pos": torch.empty(n, **i32),
                  "h_cont": torch.empty(n, d, dtype=dtype, device=dev), "out": torch.zeros(n, d, dtype=dtype, device=dev),
                  "counts": torch.empty(2, **i32)}
        self.ws = Workspace(dev)
        need = max(self.lib.tee_exit_gate_compact_scatter_workspace_size(ctypes.byref(self.gate), n),
                   fill.workspace_bytes(n))
        wp, wn = self.ws.get(need)
        t = self.t
        self.buf = StepBuffers(h_prev=t["h_prev"].data_ptr(), h_cur=t["h_cur"].data_ptr(), pos=t["pos"].data_ptr(),
                               seq=t["seq"].data_ptr(), score=t["score"].data_ptr(), mask=t["mask"].data_ptr(),
                               flag=t["flag"].data_ptr(), cont_rows=t["cont_rows"].data_ptr(),
                               exit_rows=t["exit_rows"].data_ptr(), cont_pos=t["cont_pos"].data_ptr(),
                               exit_pos=t["exit_pos"].data_ptr(), h_cont=t["h_cont"].data_ptr(),
                               out=t["out"].data_ptr(), n_out=n, counts=t["counts"].data_ptr(), ws=wp.value,
                               ws_bytes=wn)
        self.k_cache, self.v_cache = k_cache, v_cache
        self.layout = cache_layout(k_cache)
        self.handle = ctypes.c_void_p()
        st = self.lib.tee_decode_step_create(ctypes.byref(self.gate), n, ctypes.byref(fill.desc), fill.n_layers,
                                             fill.layers, _ptr(fill.prep), fill.prep.numel(), _ptr(k_cache),
                                             _ptr(v_cache), ctypes.byref(self.layout), ctypes.byref(self.buf),
                                             ctypes.byref(self.handle))
        check("tee_decode_step_create", st)
        self.stream = _stream(dev)

    def run_host(self, h_prev: torch.Tensor, h_cur: torch.Tensor, pos: torch.Tensor,
                 seq: Optional[torch.Tensor] = None, *, score: Optional[torch.Tensor] = None,
                 mask: Optional[torch.Tensor] = None, counts: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None) -> None:
        """One step: host h_prev, h_cur [n][d], pos (and seq) [n] int32 in; host score,
        mask, counts, out [n_max][d] written once the stream completes."""
        n = h_cur.shape[0]
        p = lambda t: None if t is None else t.data_ptr()   # noqa: E731 (host buffers, checked by the library)
        st = self.lib.tee_decode_step_run_host(self.handle, n, p(h_prev), p(h_cur), p(pos), p(seq), p(score), p(mask),
                                               p(counts), p(out), self.stream)
        check("tee_decode_step_run_host", st)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self.lib.tee_decode_step_destroy(h)
            self.handle = ctypes.c_void_p()


def kv_fill(h_split: torch.Tensor, layers: Sequence[Dict], k_cache: torch.Tensor, v_cache: torch.Tensor, *,
            n_kv_heads: int, head_dim: int, rope_base: float, eps: float = 1e-5, int4: bool = False,
            group: int = 64, **kw) -> KVFill:
    """One-shot convenience: prepare for these layers and fill; returns the prepared object."""
    f = KVFill(layers, d=h_split.shape[1], n_kv_heads=n_kv_heads, head_dim=head_dim, rope_base=rope_base, eps=eps,
               dtype=h_split.dtype, max_pos=k_cache.shape[3], int4=int4, group=group)
    f(h_split, k_cache, v_cache, **kw)
    return f


def ridge_fit(x: torch.Tensor, y: torch.Tensor, lam: float, *, ws: Optional[Workspace] = None,
              out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """RidgeFill's map W = (X^T X + lam I)^-1 X^T Y on the GPU: x [n][d], y [n][d_out]
    bf16 calibration rows; returns W [d][d_out] fp32."""
    lib = load()
    x = _mat(x, "x")
    _mat(y, "y")
    n, d = x.shape
    d_out = y.shape[1]
    if y.shape[0] != n:
        raise ValueError("x and y need the same rows")
    w = out if out is not None else torch.empty(d, d_out, dtype=torch.float32, device=x.device)
    ws = ws or Workspace(x.device)
    wp, wn = ws.get(lib.tee_ridge_fit_workspace_size(n, d, d_out))
    st = lib.tee_ridge_fit(n, d, d_out, _ptr(x), x.stride(0), _ptr(y), y.stride(0), _DT[x.dtype], float(lam), _ptr(w),
                           w.stride(0), wp, wn, _stream(x.device))
    check("tee_ridge_fit", st)
    return w


class ExitRiver:
    """Prepared Exit River: the W4A16 copies of the layers an exited token
    still runs (River-LLM), for a fixed set of layers and cache length.

    ``layers`` holds one dict per exit layer, in order: bf16 CUDA tensors
    ``attn_norm``, ``ffn_norm`` [d]; for each of q k v o g u d the packed int4
    codes ``w{m}`` [k_in/2][n_out] u8 and fp16 ``{m}_scale``, ``{m}_zero``
    [k_in/64][n_out]; and the int ``cache_layer``. ``attn`` forces the
    attention's walk of the cache (``"pair"`` or ``"chunk"``, see
    ``TEE_RIVER_ATTN_BY_PAIR``); ``"auto"`` picks it from the item count.
    """

    def __init__(self, layers: Sequence[Dict], *, d: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 d_ff: int, rope_base: float, eps: float, max_pos: int, group: int = 64, attn: str = "auto"):
        self.lib = load()
        flags = {"auto": 0, "pair": _lib.TEE_RIVER_ATTN_BY_PAIR, "chunk": _lib.TEE_RIVER_ATTN_BY_CHUNK}[attn]
        self.desc = _lib.RiverDesc(d=d, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim, d_ff=d_ff,
                                   rope_base=float(rope_base), eps=float(eps), group=group, flags=flags)
        self.keep: List[torch.Tensor] = []
        arr = (_lib.RiverLayer * max(1, len(layers)))()

        def p(L, k):
            t = _vec(L[k], k)
            self.keep.append(t)
            return t.data_ptr()

        dev = None
        for i, L in enumerate(layers):
            arr[i].attn_norm, arr[i].ffn_norm = p(L, "attn_norm"), p(L, "ffn_norm")
            for m in "qkvougd":
                w = getattr(arr[i], f"w{m}")
                w.codes, w.scale, w.zero = p(L, f"w{m}"), p(L, f"{m}_scale"), p(L, f"{m}_zero")
            arr[i].cache_layer = int(L["cache_layer"])
            dev = L["attn_norm"].device
        self.layers = arr
        self.n_layers = len(layers)
        self.max_pos = int(max_pos)
        self.device = dev or torch.device("cuda")
        nbytes = self.lib.tee_exit_river_prep_size(ctypes.byref(self.desc), self.n_layers, self.max_pos)
        if nbytes == 0:
            raise ValueError("invalid Exit River descriptor")
        self.prep = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        check("tee_exit_river_prepare", self.lib.tee_exit_river_prepare(
            ctypes.byref(self.desc), self.n_layers, self.layers, self.max_pos, _ptr(self.prep), nbytes,
            _stream(self.device)))

    def workspace_bytes(self, n_max: int, max_pos: Optional[int] = None) -> int:
        return self.lib.tee_exit_river_workspace_size(ctypes.byref(self.desc), int(n_max),
                                                      int(max_pos or self.max_pos))

    def __call__(self, h: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, pos: torch.Tensor, *,
                 seq: Optional[torch.Tensor] = None, rows: Optional[torch.Tensor] = None,
                 n_dev: Optional[torch.Tensor] = None, n_max: Optional[int] = None,
                 out: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None) -> torch.Tensor:
        """Runs the items through every exit layer; returns h_out [n_max][d] (bf16)."""
        _mat(h, "h")
        if k_cache.stride() != v_cache.stride() or k_cache.shape != v_cache.shape:
            raise ValueError("k_cache and v_cache must share one layout")
        layout = cache_layout(k_cache)
        if n_max is None:
            n_max = rows.numel() if rows is not None else h.shape[0]
        if out is None:
            out = torch.empty(int(n_max), h.shape[1], dtype=h.dtype, device=h.device)
        _mat(out, "out")
        ws = ws or Workspace(h.device)
        wp, wn = ws.get(self.workspace_bytes(n_max, layout.max_pos))
        st = self.lib.tee_exit_river(ctypes.byref(self.desc), self.n_layers, self.layers, _ptr(self.prep),
                                     self.prep.numel(), int(n_max), _ptr(_vec(n_dev, "n_dev")), _ptr(h), h.stride(0),
                                     h.shape[0], _ptr(_vec(rows, "rows")), _ptr(_vec(pos, "pos")),
                                     _ptr(_vec(seq, "seq")), _ptr(k_cache), _ptr(v_cache), ctypes.byref(layout),
                                     _ptr(out), out.stride(0), wp, wn, _stream(h.device))
        check("tee_exit_river", st)
        return out
