"""Oracle for the ragged n-gram hash IDs (``compute_ngram_ids``).

TEST INFRASTRUCTURE (see the package docstring).

Source: PR#54517 report ("Fuse Qwen4Exp PLE kernels"), section 关键源码片段:
  * the CPU branch of ``compute_ngram_ids`` in ``ple_layer.py`` -- every
    request gets a row pre-filled with ``eos_token_id``; token ``pos`` belongs
    to request ``searchsorted(query_start_loc, pos, right=True) - 1`` clamped to
    ``num_reqs - 1``, at column ``pos - query_start_loc[req]``;
  * the skeleton of ``_ple_ngram_ids_kernel`` in ``ops/ple.py`` -- for every
    shift 1..NGRAM_CONTEXT_LEN the prefix token comes from the request or from
    ``ngram_context``; once an EOS has been crossed every earlier token is
    replaced by EOS; the hash is an XOR mix of ``token * multiplier``, reduced
    per head into that head's partition of the table; int64 overflow behaves
    like ``torch.remainder`` on int64.

Readings taken where the pages are silent or garbled (each is listed in the
design notes of the repository as well):
  * The hash XOR-accumulates the raw wrapped int64 products and reduces only
    when a head is emitted: ``id = remainder(mixed, V_h) + O_h``. (The
    skeleton's comment fuses the mix and the reduction into one garbled line;
    reducing every term first could never overflow, yet overflow is a tested
    case.)
  * ``layer_multipliers`` has NGRAM_CONTEXT_LEN + 1 entries, indexed by the
    token's lag (0 = current token), shared by all n-gram orders.
  * Orders n = 2 .. NGRAM_CONTEXT_LEN + 1 are emitted (no unigram head); head
    ``h = (n - 2) * heads_per_ngram + j``.
  * EOS crossing: an EOS at lag j >= 1 is kept and every lag > j becomes EOS;
    the current token being EOS does not trigger it.
  * ``ngram_context[r]`` holds request r's previous NGRAM_CONTEXT_LEN tokens,
    oldest first; ``None`` means "no history" (all EOS, the EOS padding at
    request starts).
  * Tokens at or past ``query_start_loc[num_reqs]`` continue the last request
    (the clamp of the CPU branch).
"""

_INT64_MOD = 1 << 64
_INT64_HALF = 1 << 63


def wrap_int64(value):
    """Reduce a Python int to the int64 value with the same low 64 bits."""
    return ((int(value) + _INT64_HALF) % _INT64_MOD) - _INT64_HALF


def request_spans(query_start_loc, num_tokens):
    """[start, end) token span of each request.

    Token t belongs to the last request r with ``query_start_loc[r] <= t``
    (right-sided search minus one), clamped to the last request; so an empty
    request owns nothing and the last request also owns every token from its
    start up to ``num_tokens``.
    """
    qsl = [int(x) for x in query_start_loc]
    num_reqs = len(qsl) - 1
    spans = []
    for r in range(num_reqs):
        start = qsl[r]
        end = qsl[r + 1] if r + 1 < num_reqs else num_tokens
        spans.append((start, max(start, end)))
    return spans


def ngram_ids(input_ids, query_start_loc, ngram_context, layer_multipliers,
              vocab_sizes, offsets, eos_token_id, heads_per_ngram,
              num_tokens=None):
    """n-gram hash IDs of every token.

    Args:
      input_ids: flat sequence of token ids (ints), length ``num_tokens``.
      query_start_loc: request boundaries, length ``num_reqs + 1``,
        ``query_start_loc[0] == 0``, non-decreasing.
      ngram_context: ``num_reqs`` rows of NGRAM_CONTEXT_LEN previous tokens,
        oldest first, or ``None`` for fresh requests.
      layer_multipliers: NGRAM_CONTEXT_LEN + 1 int64 multipliers of this layer.
      vocab_sizes, offsets: per head V_h > 0 and O_h, heads ordered by n-gram
        order then head index.
      eos_token_id, heads_per_ngram: as named.

    Returns:
      (ids, context_out): ``ids[t][h]`` as a list of lists of Python ints, and
      each request's last NGRAM_CONTEXT_LEN tokens of its virtual sequence
      (history followed by its tokens), the carry-over for the next step.
    """
    tokens = [int(x) for x in input_ids]
    if num_tokens is None:
        num_tokens = len(tokens)
    mult = [int(m) for m in layer_multipliers]
    ctx_len = len(mult) - 1
    num_heads = ctx_len * heads_per_ngram
    V = [int(v) for v in vocab_sizes]
    O = [int(o) for o in offsets]
    assert ctx_len >= 1 and len(V) == num_heads and len(O) == num_heads
    assert all(v > 0 for v in V)
    eos = int(eos_token_id)

    ids = [[0] * num_heads for _ in range(num_tokens)]
    context_out = []
    for r, (start, end) in enumerate(request_spans(query_start_loc, num_tokens)):
        if ngram_context is None:
            history = [eos] * ctx_len
        else:
            history = [int(x) for x in ngram_context[r]]
            assert len(history) == ctx_len
        seq = history + tokens[start:end]
        for p in range(ctx_len, len(seq)):
            t = start + p - ctx_len
            lagged = [seq[p - s] for s in range(ctx_len + 1)]
            crossed = False
            for s in range(1, ctx_len + 1):
                if crossed:
                    lagged[s] = eos
                elif lagged[s] == eos:
                    crossed = True
            mixed = wrap_int64(lagged[0] * mult[0])
            for s in range(1, ctx_len + 1):
                # XOR of two values in int64 range stays in int64 range
                # (Python ints behave as infinite two's complement).
                mixed = mixed ^ wrap_int64(lagged[s] * mult[s])
                order_base = (s - 1) * heads_per_ngram
                for j in range(heads_per_ngram):
                    h = order_base + j
                    # Python % with a positive divisor is floor-mod, the
                    # semantics of torch.remainder: result in [0, V_h).
                    ids[t][h] = mixed % V[h] + O[h]
        context_out.append(seq[-ctx_len:])
    return ids, context_out
