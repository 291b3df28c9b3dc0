"""Static check of the allocation-free cache entry point: no function of the
library reachable from ``fattn_fwd_kvcache_noalloc`` names a device or host
allocation call.  The call graph is read from the C++ sources (comments
stripped): every identifier in a body that names a function defined in the
library is followed, so a new callee is covered as soon as it is written."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "exact_attention_forward_10_gb300", "csrc")
ENTRY = "fattn_fwd_kvcache_noalloc"
ALLOC = re.compile(r"\b(cudaMalloc\w*|cuMemAlloc\w*|cudaHostAlloc|cuMemHostAlloc|cuMemCreate|"
                   r"cudaMallocHost|malloc|calloc|realloc|aligned_alloc|posix_memalign)\s*\(|"
                   r"\bnew\b|\bmake_unique\b|\bmake_shared\b|\.(resize|reserve|push_back|emplace_back)\s*\(")
KEYWORDS = {"if", "for", "while", "switch", "return", "sizeof", "catch", "decltype",
            "static_assert", "alignof", "defined"}


def strip_comments(src: str) -> str:
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return re.sub(r'"(\\.|[^"\\])*"', '""', src)


def match(src: str, i: int, open_c: str, close_c: str) -> int:
    """Index just past the bracket that closes the one at ``i``."""
    depth = 0
    for j in range(i, len(src)):
        if src[j] == open_c:
            depth += 1
        elif src[j] == close_c:
            depth -= 1
            if depth == 0:
                return j + 1
    raise ValueError("unbalanced")


def definitions(src: str) -> dict:
    """name -> bodies of the functions defined in ``src`` (``name(...) {``)."""
    out = {}
    for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(", src):
        name = m.group(1)
        if name in KEYWORDS:
            continue
        try:
            close = match(src, m.end() - 1, "(", ")")
        except ValueError:
            continue
        rest = src[close:close + 200]
        h = re.match(r"\s*(const\s*)?(noexcept\s*)?(->\s*[\w:<>\s\*&]+)?\{", rest)
        if not h:
            continue
        start = close + h.end() - 1
        before = src[max(0, m.start() - 40):m.start()]
        if re.search(r"(=|\breturn|\(|,|&&|\|\||!)\s*$", before):
            continue  # a call or an expression, not a definition
        out.setdefault(name, []).append(src[start:match(src, start, "{", "}")])
    return out


def library_functions() -> dict:
    defs = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, f)) as fh:
                for k, v in definitions(strip_comments(fh.read())).items():
                    defs.setdefault(k, []).extend(v)
    return defs


def reachable(defs: dict, entry: str) -> set:
    seen, todo = set(), [entry]
    while todo:
        n = todo.pop()
        if n in seen or n not in defs:
            continue
        seen.add(n)
        for body in defs[n]:
            todo.extend(w for w in set(re.findall(r"\b[A-Za-z_]\w*\b", body)) if w in defs)
    return seen


def test_the_walk_sees_the_entry_and_its_callees():
    defs = library_functions()
    names = reachable(defs, ENTRY)
    # the set-up, the checks, the tensor maps and the launch are all followed
    for want in (ENTRY, "noalloc_device", "kvcache_checks", "check_device_buffer",
                 "encode_cache", "launch"):
        assert want in names, want


def test_nothing_reachable_allocates():
    defs = library_functions()
    bad = []
    for n in sorted(reachable(defs, ENTRY)):
        for body in defs[n]:
            for m in ALLOC.finditer(body):
                bad.append(f"{n}: {m.group(0)}")
    assert not bad, bad


def test_the_check_finds_an_allocation():
    # the same walk over a planted source that allocates two calls deep
    src = strip_comments("""
        static int helper2(int n) { void* p; cudaMalloc(&p, n); return 0; }
        int helper(int n) { return helper2(n); }
        int fattn_fwd_kvcache_noalloc(int n) { if (n) { return helper(n); } return 0; }
        int unrelated(void) { void* q = malloc(4); return q != 0; }
    """)
    defs = definitions(src)
    names = reachable(defs, ENTRY)
    assert names == {ENTRY, "helper", "helper2"}
    hits = [n for n in names for b in defs[n] if ALLOC.search(b)]
    assert hits == ["helper2"]


def test_the_workspace_entry_is_seen_to_allocate():
    # control on the real sources: the entry that keeps a per-device status
    # block reaches its one-time cudaMalloc through the same walk
    defs = library_functions()
    hits = {n for n in reachable(defs, "fattn_fwd_kvcache") for b in defs[n] if ALLOC.search(b)}
    assert "current_device" in hits
