// psk_group_run: one fusion group -- a connected chain of up to 64
// elementwise nodes sharing one loop nest -- evaluated per element in f32, the
// root alone rounded to its storage type (PSK-Realize, "What a group is";
// "What it buys": fusion reassociates nothing, only the intermediates stay in
// registers).
//
// Host side: the postfix node program is validated and compiled to a short
// accumulator-machine code (LOAD, STORE and one instruction per node) whose
// operands are per-thread value slots; inputs are loaded into the first slots,
// a node that is read again later (a REF, or an operand left below the top of
// the stack) is kept in a slot until its last read.  The code, the
// immediates and the input descriptors travel in a __grid_constant__ kernel
// parameter (the constant bank), so concurrent launches never share state.
//
// Device side: a grid-stride loop over vectors of V consecutive output
// elements along the last axis; per vector the inputs are loaded (128-bit
// or 64-bit vector loads where an input is contiguous, one load where it is
// broadcast along the last axis), then the code runs with a warp-uniform
// dispatch, the accumulator in registers and the slots in shared memory laid
// out [slot][thread] (conflict-free).  exp/erf are correctly rounded, with
// their tables staged once per CTA in shared memory.

#include <string.h>
#include <vector>

#include "common.cuh"
#include "crmath.cuh"

namespace psk {

// ------------------------------------------------------ device code format
// Instructions with an operand come first (LOAD .. MIN_R); the _R forms take
// the operand as their first argument (acc = operand OP acc).
enum : uint32_t {
  D_LOAD = 1,
  D_ADD, D_SUB, D_MUL, D_DIV, D_MAX, D_MIN,
  D_SUB_R, D_DIV_R, D_MAX_R, D_MIN_R,
  D_STORE,
  D_NEG, D_ABS, D_EXP, D_EXPC, D_GELU, D_SQRT, D_SQRTA, D_ERF,
};
constexpr uint32_t F_IMM = 1u << 8;   // operand is an immediate (else a slot)
constexpr int MAX_CODE = 3 * PSK_MAX_NODES + 8;

enum : int32_t { IN_CONTIG = 0, IN_BCAST = 1, IN_GATHER = 2 };

struct GroupInput {
  const void* ptr;
  int64_t stride[4];   // per collapsed output axis
  int32_t dtype;
  int32_t mode;        // how the last axis is read
};

struct GroupParams {
  GroupInput in[PSK_MAX_INPUTS];
  uint32_t code[MAX_CODE];
  float imm[PSK_MAX_IMM];
  void* out;
  int32_t n_in, n_code, n_slots, out_dtype;
  uint32_t rank;            // collapsed rank, 1..4 (axes padded at the front)
  uint32_t dim[4];          // collapsed dims (dim[3] = last axis)
  FastDiv div_cv;           // vectors per row: dim[3] / V
  FastDiv div2, div1;       // dim[2], dim[1]
  uint64_t v_begin;         // first vector of this launch
  uint32_t n_vec;           // vectors in this launch
};

// ---------------------------------------------------------- host compiler
struct Compiled {
  std::vector<uint32_t> code;
  int n_nodes = 0;
  int n_slots = 0;
};

static int compile_program(const psk_program* p, int n_in, Compiled& c) {
  if (!p) return fail(PSK_E_NULL, "program is NULL");
  if (p->n_tokens < 1 || p->n_tokens > PSK_MAX_TOKENS)
    return fail(PSK_E_PROGRAM, "program has %d tokens (1..%d)", p->n_tokens, PSK_MAX_TOKENS);
  if (!p->tokens) return fail(PSK_E_NULL, "program tokens are NULL");
  if (p->n_imm < 0 || p->n_imm > PSK_MAX_IMM) return fail(PSK_E_ARG, "n_imm %d (0..%d)", p->n_imm, PSK_MAX_IMM);
  if (p->n_imm > 0 && !p->imm) return fail(PSK_E_NULL, "immediates are NULL");
  if (n_in < 0 || n_in > PSK_MAX_INPUTS) return fail(PSK_E_ARG, "n_inputs %d (0..%d)", n_in, PSK_MAX_INPUTS);

  const int T = p->n_tokens;
  // Pass 1: validate and find each node's last read by REF.
  std::vector<int> last_ref;  // node -> token position of its last REF, -1 if none
  {
    int depth = 0, nodes = 0;
    for (int pos = 0; pos < T; ++pos) {
      uint32_t t = p->tokens[pos], op = t >> 24, arg = t & 0xFFFFFFu;
      switch (op) {
        case PSK_OP_IN:
          if ((int)arg >= n_in) return fail(PSK_E_PROGRAM, "token %d: input %u of %d", pos, arg, n_in);
          ++depth; break;
        case PSK_OP_IMM:
          if ((int)arg >= p->n_imm) return fail(PSK_E_PROGRAM, "token %d: immediate %u of %d", pos, arg, p->n_imm);
          ++depth; break;
        case PSK_OP_REF:
          if ((int)arg >= nodes) return fail(PSK_E_PROGRAM, "token %d: REF %u before node exists", pos, arg);
          last_ref[arg] = pos; ++depth; break;
        case PSK_OP_ADD: case PSK_OP_SUB: case PSK_OP_MUL: case PSK_OP_DIV: case PSK_OP_MAX: case PSK_OP_MIN:
          if (depth < 2) return fail(PSK_E_PROGRAM, "token %d: binary op with %d operand(s)", pos, depth);
          --depth; ++nodes; last_ref.push_back(-1); break;
        case PSK_OP_NEG: case PSK_OP_ABS: case PSK_OP_EXP: case PSK_OP_EXPC: case PSK_OP_GELU:
        case PSK_OP_SQRT: case PSK_OP_SQRTA: case PSK_OP_ERF:
          if (depth < 1) return fail(PSK_E_PROGRAM, "token %d: unary op with no operand", pos);
          ++nodes; last_ref.push_back(-1); break;
        default:
          return fail(PSK_E_PROGRAM, "token %d: unknown opcode 0x%02x", pos, op);
      }
      if (nodes > PSK_MAX_NODES)
        return fail(PSK_E_TOO_MANY_NODES, "token %d: node %d past the cap of %d", pos, nodes, PSK_MAX_NODES);
    }
    if (nodes == 0) return fail(PSK_E_PROGRAM, "program has no op node");
    if (depth != 1) return fail(PSK_E_PROGRAM, "%d values left on the stack (must be 1)", depth);
    c.n_nodes = nodes;
  }

  // Pass 2: accumulator code.  Stack entries: the accumulator, a slot or an
  // immediate.  Slots 0..n_in-1 hold the inputs; the rest are allocated for
  // spilled stack entries and REF'd nodes and freed after their last read.
  struct Ent { int kind; int idx; bool owned; };  // kind 0 acc, 1 slot, 2 imm
  std::vector<Ent> st;
  std::vector<int> free_slots;
  std::vector<int> node_slot(c.n_nodes, -1);
  int n_slots = n_in, node = 0;
  auto alloc = [&]() { if (!free_slots.empty()) { int s = free_slots.back(); free_slots.pop_back(); return s; } return n_slots++; };
  auto release = [&](const Ent& e) { if (e.kind == 1 && e.owned) free_slots.push_back(e.idx); };
  auto emit = [&](uint32_t dop, uint32_t flags, uint32_t idx) { c.code.push_back(dop | flags | (idx << 16)); };
  auto operand_flags = [&](const Ent& e) { return e.kind == 2 ? F_IMM : 0u; };
  auto spill_acc = [&]() {   // move a live accumulator entry into a slot
    for (auto& e : st) if (e.kind == 0) { int s = alloc(); emit(D_STORE, 0, s); e = Ent{1, s, true}; }
  };
  static const uint32_t bin_map[6] = {D_ADD, D_SUB, D_MUL, D_DIV, D_MAX, D_MIN};
  // reversed operand order; ADD and MUL are commutative bit for bit
  static const uint32_t rev_map[6] = {D_ADD, D_SUB_R, D_MUL, D_DIV_R, D_MAX_R, D_MIN_R};
  static const uint32_t un_map[8] = {D_NEG, D_ABS, D_EXP, D_EXPC, D_GELU, D_SQRT, D_SQRTA, D_ERF};
  // REF entries of one node share its slot; it is freed after the last REF is consumed.
  std::vector<int> ref_pending(c.n_nodes, 0);
  for (int pos = 0; pos < T; ++pos) {
    uint32_t t = p->tokens[pos], op = t >> 24, arg = t & 0xFFFFFFu;
    if (op == PSK_OP_REF) ++ref_pending[arg];
  }
  auto consume = [&](const Ent& e) {
    if (e.kind == 1 && e.owned) { release(e); return; }
    if (e.kind == 1 && e.idx >= n_in) {      // a node slot read through REF
      for (int k = 0; k < c.n_nodes; ++k)
        if (node_slot[k] == e.idx && --ref_pending[k] == 0) { free_slots.push_back(e.idx); node_slot[k] = -2; }
    }
  };
  for (int pos = 0; pos < T; ++pos) {
    uint32_t t = p->tokens[pos], op = t >> 24, arg = t & 0xFFFFFFu;
    if (op == PSK_OP_IN) { st.push_back(Ent{1, (int)arg, false}); continue; }
    if (op == PSK_OP_IMM) { st.push_back(Ent{2, (int)arg, false}); continue; }
    if (op == PSK_OP_REF) { st.push_back(Ent{1, node_slot[arg], false}); continue; }
    if (op >= PSK_OP_ADD && op <= PSK_OP_MIN) {
      Ent b = st.back(); st.pop_back();
      Ent a = st.back(); st.pop_back();
      uint32_t dop = bin_map[op - PSK_OP_ADD];
      if (a.kind == 0) {
        emit(dop, operand_flags(b), b.idx);
      } else if (b.kind == 0) {
        emit(rev_map[op - PSK_OP_ADD], operand_flags(a), a.idx);
      } else {
        spill_acc();
        emit(D_LOAD, operand_flags(a), a.idx);
        emit(dop, operand_flags(b), b.idx);
      }
      consume(a);
      consume(b);
    } else {
      Ent a = st.back(); st.pop_back();
      if (a.kind != 0) { spill_acc(); emit(D_LOAD, operand_flags(a), a.idx); }
      emit(un_map[op - PSK_OP_NEG], 0, 0);
      consume(a);
    }
    st.push_back(Ent{0, 0, false});
    if (last_ref[node] >= 0) {             // read again later through REF
      int s = alloc();
      emit(D_STORE, 0, s);
      node_slot[node] = s;
    }
    ++node;
  }
  if ((int)c.code.size() > MAX_CODE) return fail(PSK_E_PROGRAM, "compiled code too long (%zu)", c.code.size());
  c.n_slots = n_slots;
  return PSK_OK;
}

// ------------------------------------------------------------- device side
constexpr int GROUP_THREADS = 128;

struct MathTables {
  float exp_hi[32], exp_lo[32];
  float erf_hi[(PSK_ERF_D32 + 1) * 32];
  float erf_lo[PSK_ERF_NPAIR * 32];
};

__device__ __forceinline__ void load_tables(MathTables& t) {
  for (int i = threadIdx.x; i < 32; i += blockDim.x) { t.exp_hi[i] = psk_exp_tab_hi[i]; t.exp_lo[i] = psk_exp_tab_lo[i]; }
  for (int i = threadIdx.x; i < (PSK_ERF_D32 + 1) * 32; i += blockDim.x) t.erf_hi[i] = (&psk_erf_c32hi[0][0])[i];
  for (int i = threadIdx.x; i < PSK_ERF_NPAIR * 32; i += blockDim.x) t.erf_lo[i] = (&psk_erf_c32lo[0][0])[i];
}

template <int V> struct Vec { float v[V]; };

template <int V>
__device__ __forceinline__ Vec<V> load_input(const GroupInput& in, int64_t off, int64_t s_last) {
  Vec<V> r;
  if (in.dtype == PSK_F32) {
    const float* p = (const float*)in.ptr + off;
    if (V == 4 && in.mode == IN_CONTIG) {
      float4 q = __ldg((const float4*)p);
      r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[V > 3 ? 3 : 0] = q.w;
    } else if (in.mode == IN_BCAST) {
      float q = __ldg(p);
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = q;
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = __ldg(p + j * s_last);
    }
  } else {
    const uint16_t* p = (const uint16_t*)in.ptr + off;
    if (V == 4 && in.mode == IN_CONTIG) {
      uint2 q = __ldg((const uint2*)p);
      r.v[0] = __uint_as_float(q.x << 16);
      r.v[1] = __uint_as_float(q.x & 0xFFFF0000u);
      r.v[2] = __uint_as_float(q.y << 16);
      r.v[V > 3 ? 3 : 0] = __uint_as_float(q.y & 0xFFFF0000u);
    } else if (in.mode == IN_BCAST) {
      float q = bf16_bits_to_f32(__ldg(p));
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = q;
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = bf16_bits_to_f32(__ldg(p + j * s_last));
    }
  }
  return r;
}

// Unary nodes on the V accumulator lanes.  For exp and erf the tier-1 cores
// of all V elements run first (independent chains the scheduler interleaves),
// and only undecided elements go to the slower tiers.
template <int V>
__device__ __forceinline__ void op_unary(uint32_t dop, Vec<V>& acc, const MathTables& tab) {
  switch (dop) {
    case D_NEG:
#pragma unroll
      for (int j = 0; j < V; ++j) acc.v[j] = -acc.v[j];
      break;
    case D_ABS:
#pragma unroll
      for (int j = 0; j < V; ++j) acc.v[j] = fabsf(acc.v[j]);
      break;
    case D_EXP:
    case D_EXPC: {
      float a[V], R[V], d[V];
      int n[V];
      bool inr[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        a[j] = acc.v[j];
        if (dop == D_EXPC) {
          a[j] = a[j] > -4.0f ? a[j] : -4.0f;
          a[j] = a[j] < 4.0f ? a[j] : 4.0f;
        }
        inr[j] = fabsf(a[j]) <= 87.0f;
        exp_tier1_core(inr[j] ? a[j] : 0.0f, tab.exp_hi, tab.exp_lo, R[j], d[j], n[j]);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        float o = u2f((uint32_t)((int32_t)f2u(R[j]) + n[j] * (1 << 23)));
        if (!(inr[j] && tier1_decided(R[j], d[j]))) o = exp_tier2(a[j]);
        acc.v[j] = o;
      }
      break;
    }
    case D_GELU:
    case D_ERF: {
      float tt[V], R[V], d[V];
      bool inr[V];
#pragma unroll
      for (int j = 0; j < V; ++j) {
        tt[j] = dop == D_GELU ? __fmul_rn(acc.v[j], PSK_INV_SQRT2) : acc.v[j];
        const float aa = fabsf(tt[j]);
        inr[j] = aa < PSK_ERF_ONE_FROM && aa >= 0x1p-60f;
        erf_tier1_core(inr[j] ? aa : 0.5f, tab.erf_hi, tab.erf_lo, R[j], d[j]);
      }
#pragma unroll
      for (int j = 0; j < V; ++j) {
        float r = R[j];
        if (!(inr[j] && tier1_decided(R[j], d[j]))) r = erf_abs_rest(fabsf(tt[j]));
        r = copysignf(r, tt[j]);
        acc.v[j] = dop == D_GELU ? __fmul_rn(acc.v[j], __fmul_rn(0.5f, __fadd_rn(1.0f, r))) : r;
      }
      break;
    }
    case D_SQRT:
#pragma unroll
      for (int j = 0; j < V; ++j) acc.v[j] = __fsqrt_rn(acc.v[j]);
      break;
    default:  // D_SQRTA
#pragma unroll
      for (int j = 0; j < V; ++j) acc.v[j] = __fsqrt_rn(fabsf(acc.v[j]));
      break;
  }
}

template <int V, int OUT>
__global__ void __launch_bounds__(GROUP_THREADS, 4) group_kernel(const __grid_constant__ GroupParams P) {
  __shared__ MathTables tab;
  extern __shared__ float4 slot_mem[];
  load_tables(tab);
  __syncthreads();
  Vec<V>* slots = reinterpret_cast<Vec<V>*>(slot_mem);
  const int tid = threadIdx.x;
  const int bd = blockDim.x;

  for (uint32_t vi = blockIdx.x * bd + tid; vi < P.n_vec; vi += gridDim.x * bd) {
    // vector index -> (row, column vector) -> collapsed coordinates
    uint64_t v = P.v_begin + vi;
    uint32_t vlo = (uint32_t)v;   // launches never exceed 2^32 vectors in total index space per call chunk
    uint32_t row = P.div_cv.div(vlo);
    uint32_t cv = vlo - row * (P.dim[3] / V);
    uint32_t i3 = cv * V, i2 = row, i1 = 0, i0 = 0;
    if (P.rank > 2) {
      uint32_t q2 = P.div2.div(row);
      i2 = row - q2 * P.dim[2];
      if (P.rank > 3) {
        uint32_t q1 = P.div1.div(q2);
        i1 = q2 - q1 * P.dim[1];
        i0 = q1;
      } else {
        i1 = q2;
      }
    }
    for (int k = 0; k < P.n_in; ++k) {
      const GroupInput& in = P.in[k];
      int64_t off = (int64_t)i0 * in.stride[0] + (int64_t)i1 * in.stride[1] + (int64_t)i2 * in.stride[2] +
                    (int64_t)i3 * in.stride[3];
      slots[k * bd + tid] = load_input<V>(in, off, in.stride[3]);
    }
    Vec<V> acc;
#pragma unroll
    for (int j = 0; j < V; ++j) acc.v[j] = 0.0f;
    for (int pc = 0; pc < P.n_code; ++pc) {
      const uint32_t ins = P.code[pc];
      const uint32_t dop = ins & 0xFFu;
      const uint32_t idx = ins >> 16;
      Vec<V> b;
      if (dop <= D_MIN_R) {                      // the operand: a slot or an immediate
        if (ins & F_IMM) {
          const float q = P.imm[idx];
#pragma unroll
          for (int j = 0; j < V; ++j) b.v[j] = q;
        } else {
          b = slots[idx * bd + tid];
        }
      }
      switch (dop) {
        case D_LOAD: acc = b; break;
#define PSK_BIN(CASE, EXPR)                                  \
        case CASE:                                           \
          _Pragma("unroll") for (int j = 0; j < V; ++j) {    \
            const float x = acc.v[j], y = b.v[j];            \
            acc.v[j] = (EXPR);                               \
          }                                                  \
          break;
        PSK_BIN(D_ADD, __fadd_rn(x, y))
        PSK_BIN(D_SUB, __fsub_rn(x, y))
        PSK_BIN(D_MUL, __fmul_rn(x, y))
        PSK_BIN(D_DIV, __fdiv_rn(x, y))
        PSK_BIN(D_MAX, x > y ? x : y)
        PSK_BIN(D_MIN, x < y ? x : y)
        PSK_BIN(D_SUB_R, __fsub_rn(y, x))
        PSK_BIN(D_DIV_R, __fdiv_rn(y, x))
        PSK_BIN(D_MAX_R, y > x ? y : x)
        PSK_BIN(D_MIN_R, y < x ? y : x)
#undef PSK_BIN
        case D_STORE: slots[idx * bd + tid] = acc; break;
        default: op_unary<V>(dop, acc, tab); break;
      }
    }
    // root -> storage, row-major output
    uint64_t e0 = v * V;
    if (OUT == PSK_F32) {
      float* o = (float*)P.out + e0;
      if (V == 4) *(float4*)o = make_float4(acc.v[0], acc.v[1 % V], acc.v[2 % V], acc.v[3 % V]);
      else o[0] = acc.v[0];
    } else {
      uint16_t* o = (uint16_t*)P.out + e0;
      if (V == 4) {
        uint2 q;
        q.x = f32x2_to_bf16x2(acc.v[0], acc.v[1 % V]);
        q.y = f32x2_to_bf16x2(acc.v[2 % V], acc.v[3 % V]);
        *(uint2*)o = q;
      } else {
        o[0] = f32_to_bf16_bits(acc.v[0]);
      }
    }
  }
}

// ----------------------------------------------------------- host launch
template <int V, int OUT>
static int launch_group(GroupParams& P, uint64_t n_vec_total, size_t smem, cudaStream_t stream) {
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)group_kernel<V, OUT>, 200 * 1024, attr);
  int blocks_per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, group_kernel<V, OUT>, GROUP_THREADS, smem);
  if (blocks_per_sm < 1) return fail(PSK_E_SHAPE, "group needs %zu bytes of shared memory per CTA", smem);
  const uint64_t chunk = 1ull << 30;
  for (uint64_t b = 0; b < n_vec_total; b += chunk) {
    uint64_t n = n_vec_total - b < chunk ? n_vec_total - b : chunk;
    P.v_begin = b;
    P.n_vec = (uint32_t)n;
    uint64_t want = (n + GROUP_THREADS - 1) / GROUP_THREADS;
    uint64_t cap = (uint64_t)device_sm_count() * blocks_per_sm;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    group_kernel<V, OUT><<<grid, GROUP_THREADS, smem, stream>>>(P);
    int rc = check_launch("group kernel");
    if (rc) return rc;
  }
  return PSK_OK;
}

}  // namespace psk

using namespace psk;

extern "C" int psk_group_check(const psk_program* prog, int32_t n_inputs, int32_t* n_nodes, int32_t* n_slots) {
  clear_error();
  Compiled c;
  int rc = compile_program(prog, n_inputs, c);
  if (rc) return rc;
  if (n_nodes) *n_nodes = c.n_nodes;
  if (n_slots) *n_slots = c.n_slots;
  return PSK_OK;
}

extern "C" int psk_group_run(const psk_program* prog, const psk_input* inputs, int32_t n_inputs,
                             const psk_output* out, void* stream) {
  clear_error();
  Compiled c;
  int rc = compile_program(prog, n_inputs, c);
  if (rc) return rc;
  if (!out) return fail(PSK_E_NULL, "output descriptor is NULL");
  if (n_inputs > 0 && !inputs) return fail(PSK_E_NULL, "inputs are NULL");
  if (!dtype_ok(out->dtype)) return fail(PSK_E_DTYPE, "output dtype %d", out->dtype);
  if (out->rank < 0 || out->rank > PSK_MAX_RANK) return fail(PSK_E_SHAPE, "output rank %d (0..4)", out->rank);
  // shape, padded to 4 axes at the front
  int64_t shape[4] = {1, 1, 1, 1};
  uint64_t n = 1;
  for (int k = 0; k < out->rank; ++k) {
    if (out->shape[k] < 0) return fail(PSK_E_SHAPE, "output shape[%d] = %lld", k, (long long)out->shape[k]);
    shape[4 - out->rank + k] = out->shape[k];
    n *= (uint64_t)out->shape[k];
  }
  if (n == 0) return PSK_OK;  // an empty group computes nothing
  if (!out->ptr) return fail(PSK_E_NULL, "output pointer is NULL");
  for (int k = 0; k < 4; ++k)
    if (shape[k] > 0x7FFFFFFF) return fail(PSK_E_SHAPE, "axis of %lld elements (max 2^31-1)", (long long)shape[k]);

  GroupParams P;
  memset(&P, 0, sizeof(P));
  int64_t strides[PSK_MAX_INPUTS][4];
  const size_t osz = dtype_size(out->dtype);
  const char* o_lo = (const char*)out->ptr;
  const char* o_hi = o_lo + n * osz;
  for (int i = 0; i < n_inputs; ++i) {
    const psk_input& in = inputs[i];
    if (!in.ptr) return fail(PSK_E_NULL, "input %d pointer is NULL", i);
    if (!dtype_ok(in.dtype)) return fail(PSK_E_DTYPE, "input %d dtype %d", i, in.dtype);
    uint64_t span = 1;
    for (int k = 0; k < 4; ++k) strides[i][k] = 0;
    for (int k = 0; k < out->rank; ++k) {
      int64_t s = in.stride[k];
      if (s < 0) return fail(PSK_E_SHAPE, "input %d stride[%d] = %lld < 0", i, k, (long long)s);
      strides[i][4 - out->rank + k] = s;
      span += (uint64_t)s * (uint64_t)(out->shape[k] - 1);
    }
    const char* lo = (const char*)in.ptr;
    const char* hi = lo + span * dtype_size(in.dtype);
    if (lo < o_hi && o_lo < hi) {  // overlap: only the identical layout is safe
      bool same = (in.ptr == out->ptr) && (in.dtype == out->dtype);
      int64_t rs = 1;
      for (int k = 3; k >= 0 && same; --k) { if (shape[k] > 1 && strides[i][k] != rs) same = false; rs *= shape[k]; }
      if (!same) return fail(PSK_E_ALIAS, "input %d overlaps the output with another layout", i);
    }
  }
  // collapse adjacent axes that every input (and the row-major output) walks
  // as one: stride[k] == stride[k+1] * shape[k+1]
  int64_t cs[4] = {shape[0], shape[1], shape[2], shape[3]};
  int64_t cst[PSK_MAX_INPUTS][4];
  for (int i = 0; i < n_inputs; ++i) for (int k = 0; k < 4; ++k) cst[i][k] = strides[i][k];
  int rank = 4;
  for (int k = 2; k >= 0; --k) {
    bool ok = true;
    for (int i = 0; i < n_inputs && ok; ++i) ok = (cst[i][k] == cst[i][k + 1] * cs[k + 1]) || cs[k] == 1;
    if (ok && cs[k] * cs[k + 1] <= 0x7FFFFFFF) {
      // merge axis k into k+1 and shift the leading axes down
      cs[k + 1] *= cs[k];
      for (int j = k; j > 0; --j) cs[j] = cs[j - 1];
      cs[0] = 1;
      for (int i = 0; i < n_inputs; ++i) { for (int j = k; j > 0; --j) cst[i][j] = cst[i][j - 1]; cst[i][0] = 0; }
      --rank;
    }
  }
  // vector width: 4 consecutive elements along the last axis when every
  // contiguous input and the output line up on 16/8-byte boundaries
  int V = (cs[3] % 4 == 0) ? 4 : 1;
  if (V == 4 && ((uintptr_t)out->ptr % (4 * osz)) != 0) V = 1;
  for (int i = 0; i < n_inputs && V == 4; ++i) {
    if (cst[i][3] != 1) continue;
    size_t es = dtype_size(inputs[i].dtype);
    if ((uintptr_t)inputs[i].ptr % (4 * es) != 0) V = 1;
    for (int k = 0; k < 3; ++k) if (cs[k] > 1 && cst[i][k] % 4 != 0) V = 1;
  }
  for (int i = 0; i < n_inputs; ++i) {
    GroupInput& g = P.in[i];
    g.ptr = inputs[i].ptr;
    g.dtype = inputs[i].dtype;
    for (int k = 0; k < 4; ++k) g.stride[k] = cst[i][k];
    g.mode = cst[i][3] == 1 ? IN_CONTIG : (cst[i][3] == 0 ? IN_BCAST : IN_GATHER);
  }
  P.n_in = n_inputs;
  P.n_code = (int32_t)c.code.size();
  for (size_t k = 0; k < c.code.size(); ++k) P.code[k] = c.code[k];
  for (int k = 0; k < prog->n_imm; ++k) P.imm[k] = prog->imm[k];
  P.n_slots = c.n_slots;
  P.out = out->ptr;
  P.out_dtype = out->dtype;
  P.rank = (uint32_t)(rank < 1 ? 1 : rank);
  for (int k = 0; k < 4; ++k) P.dim[k] = (uint32_t)cs[k];
  P.div_cv = FastDiv((uint32_t)(cs[3] / V));
  P.div2 = FastDiv((uint32_t)cs[2]);
  P.div1 = FastDiv((uint32_t)cs[1]);
  uint64_t n_vec = n / V;
  if (n_vec >= (1ull << 32)) return fail(PSK_E_SHAPE, "%llu elements: more than 2^32 vectors", (unsigned long long)n);
  size_t smem = (size_t)c.n_slots * GROUP_THREADS * V * sizeof(float);
  cudaStream_t s = (cudaStream_t)stream;
  if (V == 4) {
    return out->dtype == PSK_F32 ? launch_group<4, PSK_F32>(P, n_vec, smem, s) : launch_group<4, PSK_BF16>(P, n_vec, smem, s);
  }
  return out->dtype == PSK_F32 ? launch_group<1, PSK_F32>(P, n_vec, smem, s) : launch_group<1, PSK_BF16>(P, n_vec, smem, s);
}
