"""ctypes binding of libspecverify.so (argument marshalling only).

Every function here checks tensor devices, dtypes and shapes, then calls the C
ABI declared in include/spec_verify.h with raw device pointers and the current
CUDA stream.  All computation happens in the library's CUDA kernels; there is
no CPU or PyTorch fallback.  Importing this module raises if the library has
not been built (see ``speculative_decoding_verify_07_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libspecverify.so")

SPEC_F32 = 0
SPEC_BF16 = 1

SPEC_OK = 0
SPEC_E_NULL = -1
SPEC_E_DIM = -2
SPEC_E_DTYPE = -3
SPEC_E_ALIGN = -4
SPEC_E_WORKSPACE = -5
SPEC_E_CUDA = -6
SPEC_E_ARCH = -7

F_MARGIN_ACCEPT = 1
F_MARGIN_DRAW = 2
F_MARGIN_TOPP = 4
F_NAN = 8
F_BAD_TOKEN = 16
F_BAD_PARAM = 32
F_RESIDUAL_EMPTY = 64
F_BAD_IDX = 128
F_TIMEOUT = 256

SPEC_MAX_V = 524288
SPEC_MAX_K = 16


class SpecError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing; build it with "
            "`python -m speculative_decoding_verify_07_gb300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [i32, i32, i32]
    lib.spec_verify_workspace_size.restype = sz
    u32 = ctypes.c_uint32
    lib.spec_verify.argtypes = [vp, i32, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_verify.restype = i32
    lib.spec_commit.argtypes = [vp, vp, vp, vp, vp, vp] + [i32] * 9 + [vp, vp]
    lib.spec_commit.restype = i32
    lib.spec_commit_swap.argtypes = [vp, vp, vp, vp, vp, vp, vp] + [i32] * 9 + [vp, vp]
    lib.spec_commit_swap.restype = i32
    lib.spec_verify_commit.argtypes = ([vp, i32, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp, vp, vp, vp, sz]
                                       + [vp] * 5 + [i32] * 7 + [vp])
    lib.spec_verify_commit.restype = i32
    lib.spec_verify_noalloc.argtypes = [vp, i32, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_noalloc.restype = i32
    lib.spec_draft_workspace_size.argtypes = [i32, i32]
    lib.spec_draft_workspace_size.restype = sz
    lib.spec_draft_sample.argtypes = [vp, i32, vp, u64, u32, u32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_draft_sample.restype = i32
    lib.spec_philox4x32_10.argtypes = [vp, u64, vp, ctypes.c_int64, vp]
    lib.spec_philox4x32_10.restype = i32
    lib.spec_status_string.argtypes = [i32]
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_version.argtypes = []
    lib.spec_version.restype = i32
    return lib


LIB = _load()
LIB_PATH = _LIB_PATH


def status_string(code: int) -> str:
    return LIB.spec_status_string(int(code)).decode()


def version() -> int:
    return int(LIB.spec_version())


def workspace_size(B: int, k: int, V: int) -> int:
    return int(LIB.spec_verify_workspace_size(int(B), int(k), int(V)))


def row_block(total_rows: int, world: int, rank: int):
    """Rows [lo, hi) of a batch of `total_rows` that rank `rank` of `world`
    verifies, as contiguous blocks (the first total_rows % world ranks take
    one row more).  The rank passes row_base = lo, so that every row draws the
    random numbers of its place in the whole batch and the shards together
    give exactly the single-call result."""
    if world < 1 or not 0 <= rank < world or total_rows < 0:
        raise ValueError(f"bad shard: {total_rows} rows, rank {rank} of {world}")
    base, extra = divmod(int(total_rows), int(world))
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_params(temperature, top_k, top_p, device) -> torch.Tensor:
    """Pack per-row (temperature, top_k, top_p) into the [B, 4] int32 layout of spec_params_t."""
    T = torch.as_tensor(temperature, dtype=torch.float32).reshape(-1)
    K = torch.as_tensor(top_k, dtype=torch.int32).reshape(-1)
    P = torch.as_tensor(top_p, dtype=torch.float32).reshape(-1)
    z = torch.zeros_like(K)
    packed = torch.stack([T.view(torch.int32), K, P.view(torch.int32), z], dim=1).contiguous()
    return packed.to(device)


class VerifyOutputs:
    def __init__(self, B: int, k: int, device):
        self.tokens = torch.empty((B, k + 1), dtype=torch.int32, device=device)
        self.accept_len = torch.empty((B,), dtype=torch.int32, device=device)
        self.logprobs = torch.empty((B, k + 1), dtype=torch.float32, device=device)
        self.alpha = torch.empty((B, max(k, 0)), dtype=torch.float32, device=device)
        self.flags = torch.empty((B,), dtype=torch.int32, device=device)   # uint32 bit pattern


def new_workspace(B: int, k: int, V: int, device) -> torch.Tensor:
    """A zero-filled workspace (the library leaves it zero-filled after each call)."""
    n = workspace_size(B, k, V)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def spec_verify(logits: torch.Tensor, draft_probs, draft_tokens, params: torch.Tensor, seed: int,
                out: VerifyOutputs | None = None, workspace: torch.Tensor | None = None,
                stream=None, row_base: int = 0) -> VerifyOutputs:
    """Run the verify step; inputs and outputs are CUDA tensors (see spec_verify.h).

    logits [B, k+1, V] float32 or bfloat16; draft_probs [B, k, V] float32;
    draft_tokens [B, k] int32; params [B, 4] int32 from make_params().
    row_base: the stream row of this batch's first row (row r draws as row
    row_base + r), so that a batch split into row blocks reproduces the
    whole batch's draws.
    """
    if logits.dim() != 3:
        raise ValueError("logits must be [B, k+1, V]")
    B, k1, V = logits.shape
    k = k1 - 1
    dev = logits.device
    if logits.dtype == torch.float32:
        dt = SPEC_F32
    elif logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    if k > 0:
        _check(draft_probs, "draft_probs", torch.float32, (B, k, V), dev)
        _check(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _check(params, "params", torch.int32, (B, 4), dev)
    if out is None:
        out = VerifyOutputs(B, k, dev)
    if workspace is None:
        workspace = new_workspace(B, k, V, dev)
    rc = LIB.spec_verify(_ptr(logits), dt, _ptr(draft_probs) if k > 0 else None,
                         _ptr(draft_tokens) if k > 0 else None, _ptr(params),
                         ctypes.c_uint64(int(seed) & (2 ** 64 - 1)),
                         ctypes.c_uint32(int(row_base) & 0xFFFFFFFF), B, k, V,
                         _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.logprobs),
                         _ptr(out.alpha) if k > 0 else None, _ptr(out.flags),
                         _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify")
    return out


def spec_verify_noalloc(logits: torch.Tensor, draft_probs, draft_tokens, params: torch.Tensor,
                        seed: int, out: VerifyOutputs | None = None, stream=None,
                        row_base: int = 0) -> VerifyOutputs:
    """spec_verify with the library's own scratch array instead of a workspace.

    For callers that cannot allocate device scratch; the library allocates
    nothing either (see spec_verify_noalloc in spec_verify.h for the size
    limit and for why overlapping calls race).  `out` may be preallocated.
    """
    if logits.dim() != 3:
        raise ValueError("logits must be [B, k+1, V]")
    B, k1, V = logits.shape
    k = k1 - 1
    dev = logits.device
    if logits.dtype == torch.float32:
        dt = SPEC_F32
    elif logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    if k > 0:
        _check(draft_probs, "draft_probs", torch.float32, (B, k, V), dev)
        _check(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _check(params, "params", torch.int32, (B, 4), dev)
    if out is None:
        out = VerifyOutputs(B, k, dev)
    rc = LIB.spec_verify_noalloc(_ptr(logits), dt, _ptr(draft_probs) if k > 0 else None,
                                 _ptr(draft_tokens) if k > 0 else None, _ptr(params),
                                 ctypes.c_uint64(int(seed) & (2 ** 64 - 1)),
                                 ctypes.c_uint32(int(row_base) & 0xFFFFFFFF), B, k, V,
                                 _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.logprobs),
                                 _ptr(out.alpha) if k > 0 else None, _ptr(out.flags), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_noalloc")
    return out


def _commit_dims(verify_rec, verify_conv, cache_rec, cache_conv):
    """(L, B, S, H, Dk, Dv, W, C, slots) of the commit buffers, checked."""
    if verify_rec is not None:
        L, B, S, H, Dk, Dv = verify_rec.shape
        slots = cache_rec.shape[1]
        if verify_rec.dtype != torch.float32 or cache_rec.dtype != torch.float32:
            raise TypeError("recurrent state must be float32")
        if tuple(cache_rec.shape) != (L, slots, H, Dk, Dv):
            raise ValueError("cache_rec shape mismatch")
    else:
        H = Dk = Dv = 1
    if verify_conv is not None:
        Lc, Bc, Sc, W, C = verify_conv.shape
        if verify_rec is None:
            L, B, S = Lc, Bc, Sc
            slots = cache_conv.shape[1]
        elif (Lc, Bc, Sc) != (L, B, S):
            raise ValueError("verify_conv and verify_rec disagree on [L, B, S]")
        if verify_conv.element_size() != 2 or cache_conv.element_size() != 2:
            raise TypeError("conv state must be a 16-bit type")
        if tuple(cache_conv.shape) != (L, slots, W, C):
            raise ValueError("cache_conv shape mismatch")
    else:
        W = C = 1
    if verify_rec is None and verify_conv is None:
        raise ValueError("nothing to commit")
    for t, nm in ((verify_rec, "verify_rec"), (verify_conv, "verify_conv"), (cache_rec, "cache_rec"),
                  (cache_conv, "cache_conv")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    return L, B, S, H, Dk, Dv, W, C, slots


def spec_commit(verify_rec, verify_conv, accept_len, cache_slot, cache_rec, cache_conv,
                flags=None, stream=None):
    """Commit accepted states (see spec_commit in spec_verify.h).

    verify_rec [L, B, S, H, Dk, Dv] float32 or None; verify_conv [L, B, S, W, C]
    16-bit (bfloat16/int16) or None; accept_len [B] int32; cache_slot [B] int32
    or None; cache_rec [L, slots, H, Dk, Dv]; cache_conv [L, slots, W, C].
    """
    L, B, S, H, Dk, Dv, W, C, slots = _commit_dims(verify_rec, verify_conv, cache_rec, cache_conv)
    dev = accept_len.device
    _check(accept_len, "accept_len", torch.int32, (B,), dev)
    if cache_slot is not None:
        _check(cache_slot, "cache_slot", torch.int32, (B,), dev)
    rc = LIB.spec_commit(_ptr(verify_rec), _ptr(verify_conv), _ptr(accept_len), _ptr(cache_slot),
                         _ptr(cache_rec), _ptr(cache_conv), L, B, S, H, Dk, Dv, W, C, slots,
                         _ptr(flags), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_commit")


def spec_verify_commit(logits: torch.Tensor, draft_probs, draft_tokens, params: torch.Tensor, seed: int,
                       verify_rec, verify_conv, cache_slot, cache_rec, cache_conv,
                       out: VerifyOutputs | None = None, workspace: torch.Tensor | None = None,
                       stream=None, row_base: int = 0) -> VerifyOutputs:
    """spec_verify and spec_commit in one launch (see spec_verify_commit in
    spec_verify.h): the verify outputs, and each row's accepted state
    copied into its cache slot; S = k + 1 states per row."""
    if logits.dim() != 3:
        raise ValueError("logits must be [B, k+1, V]")
    B, k1, V = logits.shape
    k = k1 - 1
    dev = logits.device
    if logits.dtype == torch.float32:
        dt = SPEC_F32
    elif logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    if k > 0:
        _check(draft_probs, "draft_probs", torch.float32, (B, k, V), dev)
        _check(draft_tokens, "draft_tokens", torch.int32, (B, k), dev)
    _check(params, "params", torch.int32, (B, 4), dev)
    L, Bc, S, H, Dk, Dv, W, C, slots = _commit_dims(verify_rec, verify_conv, cache_rec, cache_conv)
    if (Bc, S) != (B, k1):
        raise ValueError("state buffers must be [L, B, k+1, ...]")
    if cache_slot is not None:
        _check(cache_slot, "cache_slot", torch.int32, (B,), dev)
    if out is None:
        out = VerifyOutputs(B, k, dev)
    if workspace is None:
        workspace = new_workspace(B, k, V, dev)
    rc = LIB.spec_verify_commit(_ptr(logits), dt, _ptr(draft_probs) if k > 0 else None,
                                _ptr(draft_tokens) if k > 0 else None, _ptr(params),
                                ctypes.c_uint64(int(seed) & (2 ** 64 - 1)),
                                ctypes.c_uint32(int(row_base) & 0xFFFFFFFF), B, k, V,
                                _ptr(out.tokens), _ptr(out.accept_len), _ptr(out.logprobs),
                                _ptr(out.alpha) if k > 0 else None, _ptr(out.flags),
                                _ptr(workspace), workspace.numel(),
                                _ptr(verify_rec), _ptr(verify_conv), _ptr(cache_slot), _ptr(cache_rec),
                                _ptr(cache_conv), L, H, Dk, Dv, W, C, slots, _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_commit")
    return out


def spec_commit_swap(verify_rec, verify_conv, accept_len, slot_of_row, scratch_slot, cache_rec, cache_conv,
                     flags=None, stream=None):
    """Zero-copy commit (see spec_commit_swap in spec_verify.h).

    verify_rec [L, B, S-1, H, Dk, Dv] float32 or None; verify_conv [L, B, S-1, W, C]
    16-bit or None: the first S - 1 states of each row; the last state of row
    r is already in cache slot scratch_slot[r].  slot_of_row and scratch_slot
    [B] int32 are updated in place (a fully accepted row trades them).
    """
    ref = verify_rec if verify_rec is not None else verify_conv
    if ref is None:
        raise ValueError("nothing to commit")
    L, B, Sm1 = ref.shape[:3]
    S = Sm1 + 1
    if verify_rec is not None:
        _, _, _, H, Dk, Dv = verify_rec.shape
        slots = cache_rec.shape[1]
        if verify_rec.dtype != torch.float32 or cache_rec.dtype != torch.float32:
            raise TypeError("recurrent state must be float32")
        if tuple(cache_rec.shape) != (L, slots, H, Dk, Dv):
            raise ValueError("cache_rec shape mismatch")
    else:
        H = Dk = Dv = 1
    if verify_conv is not None:
        _, _, _, W, C = verify_conv.shape
        if verify_rec is None:
            slots = cache_conv.shape[1]
        if tuple(verify_conv.shape[:3]) != (L, B, Sm1):
            raise ValueError("verify_conv and verify_rec disagree on [L, B, S-1]")
        if verify_conv.element_size() != 2 or cache_conv.element_size() != 2:
            raise TypeError("conv state must be a 16-bit type")
        if tuple(cache_conv.shape) != (L, slots, W, C):
            raise ValueError("cache_conv shape mismatch")
    else:
        W = C = 1
    for t, nm in ((verify_rec, "verify_rec"), (verify_conv, "verify_conv"), (cache_rec, "cache_rec"),
                  (cache_conv, "cache_conv")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{nm} must be contiguous")
    dev = accept_len.device
    _check(accept_len, "accept_len", torch.int32, (B,), dev)
    _check(slot_of_row, "slot_of_row", torch.int32, (B,), dev)
    _check(scratch_slot, "scratch_slot", torch.int32, (B,), dev)
    rc = LIB.spec_commit_swap(_ptr(verify_rec), _ptr(verify_conv), _ptr(accept_len), _ptr(slot_of_row),
                              _ptr(scratch_slot), _ptr(cache_rec), _ptr(cache_conv), L, B, S, H, Dk, Dv, W, C,
                              slots, _ptr(flags), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_commit_swap")


class DraftOutputs:
    def __init__(self, B: int, V: int, device, with_q: bool = True):
        self.q = torch.empty((B, V), dtype=torch.float32, device=device) if with_q else None
        self.tokens = torch.empty((B,), dtype=torch.int32, device=device)
        self.logprobs = torch.empty((B,), dtype=torch.float32, device=device)
        self.flags = torch.empty((B,), dtype=torch.int32, device=device)   # uint32 bit pattern


def draft_workspace_size(B: int, V: int) -> int:
    return int(LIB.spec_draft_workspace_size(int(B), int(V)))


def new_draft_workspace(B: int, V: int, device) -> torch.Tensor:
    """A zero-filled workspace for spec_draft_sample."""
    return torch.zeros(max(draft_workspace_size(B, V), 16), dtype=torch.uint8, device=device)


def spec_draft_sample(logits: torch.Tensor, params: torch.Tensor, seed: int, pos: int,
                      out: DraftOutputs | None = None, workspace: torch.Tensor | None = None,
                      stream=None, row_base: int = 0, with_q: bool = True) -> DraftOutputs:
    """One draft step (see spec_draft_sample in spec_verify.h): logits [B, V]
    float32 or bfloat16, params [B, 4] int32 from make_params(); draws x ~ q
    and writes q (unless with_q is False)."""
    if logits.dim() != 2:
        raise ValueError("logits must be [B, V]")
    B, V = logits.shape
    dev = logits.device
    if logits.dtype == torch.float32:
        dt = SPEC_F32
    elif logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    _check(params, "params", torch.int32, (B, 4), dev)
    if out is None:
        out = DraftOutputs(B, V, dev, with_q)
    if out.q is not None:
        _check(out.q, "q", torch.float32, (B, V), dev)
    if workspace is None:
        workspace = new_draft_workspace(B, V, dev)
    rc = LIB.spec_draft_sample(_ptr(logits), dt, _ptr(params), ctypes.c_uint64(int(seed) & (2 ** 64 - 1)),
                               ctypes.c_uint32(int(row_base) & 0xFFFFFFFF), ctypes.c_uint32(int(pos) & 0xFFFFFFFF),
                               B, V, _ptr(out.q), _ptr(out.tokens), _ptr(out.logprobs), _ptr(out.flags),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_draft_sample")
    return out


def philox4x32_10(ctr: torch.Tensor, seed: int, stream=None) -> torch.Tensor:
    """Device Philox4x32-10 of a [n, 4] int32 (bit pattern) counter tensor."""
    if ctr.dim() != 2 or ctr.shape[1] != 4 or ctr.dtype != torch.int32 or not ctr.is_contiguous():
        raise ValueError("ctr must be a contiguous [n, 4] int32 tensor")
    out = torch.empty_like(ctr)
    rc = LIB.spec_philox4x32_10(_ptr(ctr), ctypes.c_uint64(int(seed) & (2 ** 64 - 1)), _ptr(out),
                                ctr.shape[0], _stream(stream))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_philox4x32_10")
    return out
