"""Torch-facing binding of the C ABI: argument marshalling only.

Each function takes torch tensors, allocates the outputs (and the
workspace) on the logits' device unless they are passed in, and calls the
C entry point of the same name on the current CUDA stream. Every step of
verification runs in the library's CUDA kernels. Host (CPU) inputs are
copied to ``device`` first; that is the end-to-end path a caller with host
buffers uses.
"""

from __future__ import annotations

from typing import Dict, Optional

import torch

from . import _lib
from ._lib import SPEC_BF16, SPEC_F32, check


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, device, dtype=None) -> torch.Tensor:
    if t.is_cuda and (dtype is None or t.dtype == dtype) and t.is_contiguous():
        return t  # the common case, kept cheap: small batches are bound by this host path
    if not t.is_cuda:
        t = t.to(device, non_blocking=True)
    if dtype is not None and t.dtype != dtype:
        t = t.to(dtype)
    return t.contiguous()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None:  # the current stream's handle without building a Stream object
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(B: int, K: int, V: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32)
    return int(_lib.load().spec_workspace_bytes(B, K, V, code))


def warped_workspace_bytes(B: int, K: int, V: int, dtype) -> int:
    """Workspace with room for the stats pass's lane records (half-lane
    maxima), which let spec_verify_chain_warped select top-k sets without a
    second pass over the rows (workspace_bytes suffices, but is slower)."""
    code = dtype if isinstance(dtype, int) else (SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32)
    return int(_lib.load().spec_warped_workspace_bytes(B, K, V, code))


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Device workspace with a 256-byte aligned start."""
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off: off + nbytes]


def spec_verify_chain(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                      out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                      device="cuda", stream=None, stats: bool = True) -> Dict[str, torch.Tensor]:
    """Chain verification (sampling at T > 0, greedy at T == 0).

    target_logits [B, K+1, V], draft_logits [B, K, V] (bf16 or fp32),
    draft_tokens [B, K] int32, u_accept [B, K] fp32, u_resample [B] fp32.
    Returns accept_len, out_tokens, row_status and (with ``stats``)
    lse_target, lse_draft, p_at_x, q_at_x."""
    lib = _lib.load()
    dev = target_logits.device if target_logits.is_cuda else torch.device(device)
    Lp = _dev(target_logits, dev)
    Lq = _dev(draft_logits, dev)
    x = _dev(draft_tokens, dev, torch.int32)
    ua = _dev(u_accept, dev, torch.float32)
    ur = _dev(u_resample, dev, torch.float32)
    B, K1, V = Lp.shape
    K = K1 - 1
    dt = _dtype_code(Lp)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
        if stats:
            out.update(lse_target=torch.empty(B, K + 1, device=dev), lse_draft=torch.empty(B, K, device=dev),
                       p_at_x=torch.empty(B, K, device=dev), q_at_x=torch.empty(B, K, device=dev))
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(B, K, V, dt), dev)
    rc = lib.spec_verify_chain(
        Lp.data_ptr(), Lq.data_ptr(), dt, x.data_ptr(), ua.data_ptr(), ur.data_ptr(), float(temperature), B, K, V,
        out["accept_len"].data_ptr(), out["out_tokens"].data_ptr(), _ptr(out.get("lse_target")),
        _ptr(out.get("lse_draft")), _ptr(out.get("p_at_x")), _ptr(out.get("q_at_x")), out["row_status"].data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream(stream))
    check("spec_verify_chain", rc)
    return out


def _prepared_inputs(target_logits, draft_logits, draft_tokens, u_accept, u_resample):
    """The prepared call's inputs exactly as the caller holds them: the
    pointers baked into the call must be the caller's own buffers, or later
    refills would go unseen. Nothing is converted or copied; anything else is
    refused."""
    named = (("target_logits", target_logits), ("draft_logits", draft_logits), ("draft_tokens", draft_tokens),
             ("u_accept", u_accept), ("u_resample", u_resample))
    for name, t in named:
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name}: a torch tensor is required")
    if target_logits.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"target_logits: bfloat16 or float32 required, got {target_logits.dtype}")
    want = dict(draft_logits=target_logits.dtype, draft_tokens=torch.int32, u_accept=torch.float32,
                u_resample=torch.float32)
    for name, t in named[1:]:
        if t.dtype != want[name]:
            raise ValueError(f"{name}: {want[name]} required, got {t.dtype} (it is not converted: the prepared "
                             f"call must read the caller's own buffer)")
    if target_logits.dim() != 3:
        raise ValueError(f"target_logits must be [B, K+1, V], got {tuple(target_logits.shape)}")
    B, K1, V = target_logits.shape
    K = K1 - 1
    shapes = dict(draft_logits=(B, K, V), draft_tokens=(B, K), u_accept=(B, K), u_resample=(B,))
    for name, t in named[1:]:
        if tuple(t.shape) != shapes[name]:
            raise ValueError(f"{name} must be {list(shapes[name])}, got {list(t.shape)}")
    for name, t in named:
        if not t.is_contiguous():
            raise ValueError(f"{name}: a contiguous tensor is required (a strided view is not copied)")
    dev = target_logits.device
    for name, t in named:
        if t.device.type != "cuda" or t.device != dev:
            raise ValueError(f"{name}: a CUDA tensor on {dev} is required, got {t.device}")
    return B, K, V


def prepare_verify_chain(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                         out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                         stats: bool = False):
    """spec_verify_chain on fixed device buffers, for a serving loop that
    refills the same tensors every step: the checks and the argument
    marshalling happen once here, and the returned function enqueues one
    verification on the current stream (or on the stream it is given) and
    returns ``out``. The inputs must be contiguous CUDA tensors on one device
    with the call's dtypes (bf16 or fp32 logits of one dtype, int32 tokens,
    fp32 uniforms): the call keeps their addresses, so a tensor that would
    need a conversion is refused (ValueError) rather than silently replaced
    by a copy. The tensors must stay alive and keep their shapes; their
    contents may change between calls."""
    B, K, V = _prepared_inputs(target_logits, draft_logits, draft_tokens, u_accept, u_resample)
    lib = _lib.load()
    dev = target_logits.device
    Lp = target_logits
    dt = _dtype_code(Lp)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
        if stats:
            out.update(lse_target=torch.empty(B, K + 1, device=dev), lse_draft=torch.empty(B, K, device=dev),
                       p_at_x=torch.empty(B, K, device=dev), q_at_x=torch.empty(B, K, device=dev))
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(B, K, V, dt), dev)
    fn = lib.spec_verify_chain
    head = (Lp.data_ptr(), draft_logits.data_ptr(), dt, draft_tokens.data_ptr(), u_accept.data_ptr(),
            u_resample.data_ptr(), float(temperature), B, K, V, out["accept_len"].data_ptr(),
            out["out_tokens"].data_ptr(), _ptr(out.get("lse_target")), _ptr(out.get("lse_draft")),
            _ptr(out.get("p_at_x")), _ptr(out.get("q_at_x")), out["row_status"].data_ptr(), workspace.data_ptr(),
            workspace.numel())
    # the buffers the pointers refer to stay alive with the function
    keep = (target_logits, draft_logits, draft_tokens, u_accept, u_resample, workspace)
    index = dev.index if dev.index is not None else torch.cuda.current_device()

    def call(stream=None):
        rc = fn(*head, _raw_stream(index) if stream is None and _raw_stream is not None else _stream(stream))
        if rc:
            check("spec_verify_chain", rc)
        return out

    call.buffers = keep
    return call


def host_workspace_bytes(B: int, K: int, V: int, dtype) -> int:
    """Device workspace for spec_verify_chain_host (staged inputs and
    outputs plus the verification workspace)."""
    code = dtype if isinstance(dtype, int) else _dtype_code(torch.empty(0, dtype=dtype))
    return int(_lib.load().spec_host_workspace_bytes(B, K, V, code))


def _host(t: torch.Tensor, name: str, dtype=None) -> torch.Tensor:
    if t.device.type != "cpu" or not t.is_contiguous() or (dtype is not None and t.dtype != dtype):
        raise ValueError(f"{name}: a contiguous CPU tensor{'' if dtype is None else f' of {dtype}'} is required")
    return t


def spec_verify_chain_host(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                           out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                           device="cuda", stream=None, synchronize: bool = True) -> Dict[str, torch.Tensor]:
    """Chain verification from host (CPU) tensors through
    spec_verify_chain_host: the library copies the inputs to the device,
    verifies and copies accept_len, out_tokens and row_status back into host
    tensors (pinned, allocated unless ``out`` holds them). Inputs: contiguous
    CPU tensors as spec_verify_chain takes them (pinned memory makes the
    copies asynchronous). With ``synchronize`` the stream is synchronised
    before returning; otherwise the caller synchronises it before reading the
    outputs and keeps the inputs alive until then."""
    lib = _lib.load()
    dev = torch.device(device)
    Lp = _host(target_logits, "target_logits")
    dt = _dtype_code(Lp)
    B, K1, V = Lp.shape
    K = K1 - 1
    sampling = float(temperature) != 0.0
    Lq = _host(draft_logits, "draft_logits", Lp.dtype) if sampling else None
    x = _host(draft_tokens, "draft_tokens", torch.int32)
    ua = _host(u_accept, "u_accept", torch.float32) if sampling else None
    ur = _host(u_resample, "u_resample", torch.float32) if sampling else None
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, pin_memory=True),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, pin_memory=True),
                   row_status=torch.empty(B, dtype=torch.int32, pin_memory=True))
    if workspace is None:
        workspace = alloc_workspace(host_workspace_bytes(B, K, V, dt), dev)
    st = _stream(stream)
    rc = lib.spec_verify_chain_host(
        Lp.data_ptr(), _ptr(Lq), dt, x.data_ptr(), _ptr(ua), _ptr(ur), float(temperature), B, K, V,
        out["accept_len"].data_ptr(), out["out_tokens"].data_ptr(), out["row_status"].data_ptr(),
        workspace.data_ptr(), workspace.numel(), st)
    check("spec_verify_chain_host", rc)
    if synchronize:
        if stream is None:
            torch.cuda.current_stream(dev).synchronize()
        elif hasattr(stream, "synchronize"):
            stream.synchronize()
        else:
            torch.cuda.ExternalStream(st).synchronize()
    return out


def _stage(name, target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
           out: Dict[str, torch.Tensor], workspace: torch.Tensor, stream=None) -> None:
    B, K1, V = target_logits.shape
    fn = getattr(_lib.load(), name)
    rc = fn(target_logits.data_ptr(), draft_logits.data_ptr(), _dtype_code(target_logits), draft_tokens.data_ptr(),
            u_accept.data_ptr(), u_resample.data_ptr(), float(temperature), B, K1 - 1, V, out["accept_len"].data_ptr(),
            out["out_tokens"].data_ptr(), _ptr(out.get("lse_target")), _ptr(out.get("lse_draft")),
            _ptr(out.get("p_at_x")), _ptr(out.get("q_at_x")), out["row_status"].data_ptr(), workspace.data_ptr(),
            workspace.numel(), _stream(stream))
    check(name, rc)


def spec_chain_scan(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                    out: Dict[str, torch.Tensor], workspace: torch.Tensor, stream=None) -> None:
    """Stage A only: streaming pass, normalisers and the acceptance decision
    (device tensors, outputs preallocated as spec_verify_chain returns them)."""
    _stage("spec_chain_scan", target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature, out,
           workspace, stream)


def spec_chain_sample(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                      out: Dict[str, torch.Tensor], workspace: torch.Tensor, stream=None) -> None:
    """Stage B only: the residual / bonus draw (after spec_chain_scan)."""
    _stage("spec_chain_sample", target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature, out,
           workspace, stream)


def spec_verify_chain_greedy(target_logits, draft_tokens, out: Optional[Dict[str, torch.Tensor]] = None,
                             workspace: Optional[torch.Tensor] = None, device="cuda",
                             stream=None) -> Dict[str, torch.Tensor]:
    """Greedy chain verification: accept_len, out_tokens, argmax_ids, row_status."""
    lib = _lib.load()
    dev = target_logits.device if target_logits.is_cuda else torch.device(device)
    Lp = _dev(target_logits, dev)
    x = _dev(draft_tokens, dev, torch.int32)
    B, K1, V = Lp.shape
    K = K1 - 1
    dt = _dtype_code(Lp)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   argmax_ids=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(B, K, V, dt), dev)
    rc = lib.spec_verify_chain_greedy(Lp.data_ptr(), dt, x.data_ptr(), B, K, V, out["accept_len"].data_ptr(),
                                      out["out_tokens"].data_ptr(), _ptr(out.get("argmax_ids")),
                                      out["row_status"].data_ptr(), workspace.data_ptr(), workspace.numel(),
                                      _stream(stream))
    check("spec_verify_chain_greedy", rc)
    return out


def spec_verify_tree_greedy(node_logits, node_tokens, retrieve_indices, n1: int, tree_mask=None,
                            out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                            device="cuda", stream=None) -> Dict[str, torch.Tensor]:
    """Merged-tree greedy verification: accept_len, best_row, path_nodes,
    out_tokens, subtree, row_status."""
    lib = _lib.load()
    dev = node_logits.device if node_logits.device.type == "cuda" else torch.device(device)
    Lt = _dev(node_logits, dev)
    tok = _dev(node_tokens, dev, torch.int32)
    R = _dev(retrieve_indices, dev, torch.int32)
    mask = None if tree_mask is None else _dev(tree_mask, dev, torch.uint8)
    B, N, V = Lt.shape
    Rn, D = R.shape[1], R.shape[2]
    dt = _dtype_code(Lt)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   best_row=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty(B, D, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, D, dtype=torch.int32, device=dev),
                   subtree=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(B, N - 1, V, dt), dev)
    rc = lib.spec_verify_tree_greedy(Lt.data_ptr(), dt, tok.data_ptr(), R.data_ptr(), _ptr(mask), B, N, Rn, D, V,
                                     int(n1), out["accept_len"].data_ptr(), out["best_row"].data_ptr(),
                                     out["path_nodes"].data_ptr(), out["out_tokens"].data_ptr(),
                                     out["subtree"].data_ptr(), out["row_status"].data_ptr(), workspace.data_ptr(),
                                     workspace.numel(), _stream(stream))
    check("spec_verify_tree_greedy", rc)
    return out


def spec_tree_confidence(node_conf, n1: int, out: Optional[Dict[str, torch.Tensor]] = None, device="cuda",
                         stream=None) -> Dict[str, torch.Tensor]:
    """Confidence routing: scores [B, 2] and choice [B] (1 or 2)."""
    lib = _lib.load()
    dev = node_conf.device if node_conf.device.type == "cuda" else torch.device(device)
    c = _dev(node_conf, dev, torch.float32)
    B, N = c.shape
    if out is None:
        out = dict(scores=torch.empty(B, 2, device=dev), choice=torch.empty(B, dtype=torch.int32, device=dev))
    rc = lib.spec_tree_confidence(c.data_ptr(), B, N, int(n1), out["scores"].data_ptr(), out["choice"].data_ptr(),
                                  _stream(stream))
    check("spec_tree_confidence", rc)
    return out


def spec_kv_compact(kv: torch.Tensor, base_pos, accept_len, path=None, out: Optional[Dict[str, torch.Tensor]] = None,
                    stream=None) -> Dict[str, torch.Tensor]:
    """KV-cache compaction after verification, in place on ``kv``.

    kv: a CUDA tensor viewed as [planes, B, S, W] (any strides, last dimension
    contiguous), for example a [layers * 2, B, S, heads * head_dim] cache.
    base_pos [B] int32: position of node 0; accept_len [B] int32 and path
    [B, D] int32 (None for chain verification) as returned by the
    verification call. Returns new_len [B] and row_status [B]."""
    lib = _lib.load()
    if kv.device.type != "cuda":
        raise ValueError("kv must be a CUDA tensor (it is compacted in place)")
    if kv.dim() != 4 or kv.stride(3) != 1:
        raise ValueError("kv must be viewed as [planes, B, S, W] with a contiguous last dimension")
    P_, B, S, W = kv.shape
    sp, sb, ss, _ = kv.stride()
    dev = kv.device
    base = _dev(torch.as_tensor(base_pos), dev, torch.int32)
    acc = _dev(torch.as_tensor(accept_len), dev, torch.int32)
    pth = None if path is None else _dev(torch.as_tensor(path), dev, torch.int32)
    if out is None:
        out = dict(new_len=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    D = 0 if pth is None else pth.shape[1]
    check("spec_kv_compact", lib.spec_kv_compact(kv.data_ptr(), kv.element_size(), P_, B, S, W, sp, sb, ss,
                                                 _ptr(base), _ptr(pth), D, _ptr(acc), _ptr(out["new_len"]),
                                                 _ptr(out["row_status"]), _stream(stream)))
    return out


def spec_tree_entropy(draft_logits, n1: int, temperature: float = 1.0, out: Optional[Dict[str, torch.Tensor]] = None,
                      workspace: Optional[torch.Tensor] = None, device="cuda", stream=None,
                      node_entropy: bool = True) -> Dict[str, torch.Tensor]:
    """Entropy routing over merged drafter trees: draft_logits [B, N, V]
    (bf16 or fp32). Returns scores [B, 2], choice [B], row_status [B] and
    (with ``node_entropy``) the per-node entropies [B, N]."""
    lib = _lib.load()
    dev = draft_logits.device if draft_logits.device.type == "cuda" else torch.device(device)
    Ld = _dev(draft_logits, dev)
    B, N, V = Ld.shape
    code = _dtype_code(Ld)
    if workspace is None:
        workspace = alloc_workspace(workspace_bytes(B, N, V, code), dev)
    if out is None:
        out = dict(scores=torch.empty(B, 2, dtype=torch.float32, device=dev),
                   choice=torch.empty(B, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
        if node_entropy:
            out["node_entropy"] = torch.empty(B, N, dtype=torch.float32, device=dev)
    check("spec_tree_entropy", lib.spec_tree_entropy(Ld.data_ptr(), code, float(temperature), B, N, V, int(n1),
                                                     _ptr(out.get("node_entropy")), _ptr(out["scores"]),
                                                     _ptr(out["choice"]), _ptr(out["row_status"]),
                                                     workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def spec_tree_expand(draft_logits, logc, M: int, temperature: float = 1.0,
                     out: Optional[Dict[str, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None,
                     device="cuda", stream=None) -> Dict[str, torch.Tensor]:
    """One drafter-tree expansion step by cumulative probability:
    draft_logits [B, F, V] (bf16 or fp32) at the F frontier nodes, logc [B, F]
    their paths' log cumulative probabilities. Returns the M best children
    as parent, token [B, M] int32, score [B, M] fp32 and row_status [B]."""
    lib = _lib.load()
    dev = draft_logits.device if draft_logits.device.type == "cuda" else torch.device(device)
    Ld = _dev(draft_logits, dev)
    B, F, V = Ld.shape
    lc = _dev(logc, dev, torch.float32)
    if tuple(lc.shape) != (B, F):
        raise ValueError(f"logc must be [{B}, {F}], got {tuple(lc.shape)}")
    code = _dtype_code(Ld)
    if workspace is None:
        need = lib.spec_expand_workspace_bytes(B, F, V, int(M), code)
        if need == 0:
            check("spec_expand_workspace_bytes", _lib.SPEC_ERR_UNSUPPORTED)
        workspace = alloc_workspace(need, dev)
    if out is None:
        out = dict(parent=torch.empty(B, M, dtype=torch.int32, device=dev),
                   token=torch.empty(B, M, dtype=torch.int32, device=dev),
                   score=torch.empty(B, M, dtype=torch.float32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev))
    check("spec_tree_expand", lib.spec_tree_expand(Ld.data_ptr(), code, float(temperature), lc.data_ptr(), B, F, V,
                                                   int(M), out["parent"].data_ptr(), out["token"].data_ptr(),
                                                   out["score"].data_ptr(), out["row_status"].data_ptr(),
                                                   workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return out


def spec_merge_trees(tokens1, mask1, retrieve1, pos1, tokens2, mask2, retrieve2, pos2, device="cuda",
                     stream=None) -> Dict[str, torch.Tensor]:
    """Merge B pairs of drafter trees under one shared root on the device.

    tokens* [B, n+1] int32, mask* [B, n+1, n+1] uint8, retrieve* [B, R, D]
    int32, pos* [B, n+1] int32. Returns tokens [B, N], mask [B, N, N],
    retrieve [B, R1+R2, max(D1, D2)], pos [B, N] and n1."""
    lib = _lib.load()
    dev = tokens1.device if tokens1.device.type == "cuda" else torch.device(device)
    t1, t2 = _dev(tokens1, dev, torch.int32), _dev(tokens2, dev, torch.int32)
    m1, m2 = _dev(mask1, dev, torch.uint8), _dev(mask2, dev, torch.uint8)
    r1, r2 = _dev(retrieve1, dev, torch.int32), _dev(retrieve2, dev, torch.int32)
    p1, p2 = _dev(pos1, dev, torch.int32), _dev(pos2, dev, torch.int32)
    B, n1, n2 = t1.shape[0], t1.shape[1] - 1, t2.shape[1] - 1
    N, (R1, D1), (R2, D2) = n1 + n2 + 1, r1.shape[1:], r2.shape[1:]
    D = max(D1, D2)
    out = dict(tokens=torch.empty(B, N, dtype=torch.int32, device=dev),
               mask=torch.empty(B, N, N, dtype=torch.uint8, device=dev),
               retrieve=torch.empty(B, R1 + R2, D, dtype=torch.int32, device=dev),
               pos=torch.empty(B, N, dtype=torch.int32, device=dev))
    check("spec_merge_trees", lib.spec_merge_trees(_ptr(t1), _ptr(m1), _ptr(r1) if R1 else None, _ptr(p1), _ptr(t2),
                                                   _ptr(m2), _ptr(r2) if R2 else None, _ptr(p2), B, n1, n2, R1, D1,
                                                   R2, D2, _ptr(out["tokens"]), _ptr(out["mask"]),
                                                   _ptr(out["retrieve"]), _ptr(out["pos"]), _stream(stream)))
    out["n1"] = n1
    return out


def spec_verify_chain_warped(target_logits, draft_logits, draft_tokens, u_accept, u_resample, temperature: float,
                             top_k: int = 0, top_p: float = 1.0, out: Optional[Dict[str, torch.Tensor]] = None,
                             workspace: Optional[torch.Tensor] = None, device="cuda",
                             stream=None) -> Dict[str, torch.Tensor]:
    """Chain verification with top-k / top-p applied to p and q (0 and 1.0:
    off). Returns accept_len, out_tokens, row_status, p_at_x, q_at_x."""
    lib = _lib.load()
    dev = target_logits.device if target_logits.is_cuda else torch.device(device)
    Lp, Lq = _dev(target_logits, dev), _dev(draft_logits, dev)
    B, K1, V = Lp.shape
    K = K1 - 1
    x = _dev(draft_tokens, dev, torch.int32)
    ua = _dev(u_accept, dev, torch.float32)
    ur = _dev(u_resample, dev, torch.float32)
    code = _dtype_code(Lp)
    if workspace is None:
        workspace = alloc_workspace(warped_workspace_bytes(B, K, V, code), dev)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
                   row_status=torch.empty(B, dtype=torch.int32, device=dev),
                   p_at_x=torch.empty(B, K, dtype=torch.float32, device=dev),
                   q_at_x=torch.empty(B, K, dtype=torch.float32, device=dev))
    check("spec_verify_chain_warped",
          lib.spec_verify_chain_warped(Lp.data_ptr(), Lq.data_ptr(), code, _ptr(x), _ptr(ua), _ptr(ur),
                                       float(temperature), int(top_k), float(top_p), B, K, V,
                                       _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out.get("p_at_x")),
                                       _ptr(out.get("q_at_x")), _ptr(out["row_status"]), workspace.data_ptr(),
                                       workspace.numel(), _stream(stream)))
    return out
